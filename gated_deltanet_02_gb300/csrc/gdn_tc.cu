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
//
// Persistent: one CTA per SM walks the chunks (batch, head, chunk) w =
// blockIdx.x, + gridDim.x, ..., heads fastest, and its warps form a pipeline
// over consecutive chunks:
//   warp 0       TMA: the chunk's raw q, k, v rows (64 x 3 x 128 bf16, rows
//                past T zero-filled) into a 2-stage ring;
//   warp 1       MMA issuer (one thread): K'K'^T of a chunk once its front
//                end is done, W = T diag(beta gamma) K' and U~ = T diag(beta) V'
//                of a chunk once its inverse is done;
//   warps 2-7    front end: conv, L2 norm, bf16; Q' rows straight to global
//                memory, K' and V' tiles into a 2-stage ring (K' also to global
//                memory), the chunk's gates;
//   warps 8-11   A = strict_lower(diag(beta) (K'K'^T * D)) from tensor
//                memory, T = (I + A)^-1 in 32 x 32 blocks (the diagonal blocks
//                by forward substitution, lane = column; T10 = -T11 A10 T00);
//   warps 12-15  T diag(beta gamma) and T diag(beta) as bf16 hi / lo tiles, then
//                W (bf16) and U~ (fp32) from tensor memory to global memory.

constexpr int kPrepThreads = 512;  // 16 warps
constexpr int kFeWarp0 = 2, kFeWarps = 6, kInvWarp0 = 8, kEpiWarp0 = 12;
static_assert(kInvWarp0 % 4 == 0 && kEpiWarp0 % 4 == 0, "a warpgroup per role covers the four TMEM lane quarters");
constexpr int kBlk = 32;                               // the inverse works on 32 x 32 blocks
constexpr int kLd = kBlk + 4;                          // fp32 block rows padded to 36 (16-byte aligned)
constexpr uint32_t kBlkBytes = kBlk * kLd * 4;
constexpr uint32_t kRawBytes = 3 * 16384;              // q, k, v: two swizzled 8 KiB column blocks each
constexpr uint32_t kPrepTile = 16384;                  // K' or V': two swizzled 8 KiB column blocks
constexpr uint32_t kOffRaw = 0;                        // [2][q | k | v]
constexpr int kPrepSlots = 3;                          // K' / V' ring depth
constexpr uint32_t kOffPrep = kOffRaw + 2 * kRawBytes;  // [3][K' | V']
constexpr uint32_t kOffPG = kOffPrep + kPrepSlots * 2 * kPrepTile;  // [3][g2[64] | beta[64]]
constexpr uint32_t kOffAT = kOffPG + kPrepSlots * 512;  // A00^T, A10, A11^T, T00, T10, T11 (X reuses A00^T)
constexpr uint32_t kOffCol = kOffAT + 6 * kBlkBytes;   // [2][beta_k 2^g_k [64], beta_k [64]]
constexpr uint32_t kOffPBar = kOffCol + 1024;
constexpr uint32_t kPrepSmem = kOffPBar + 256 + 1024;
static_assert(kOffPrep % 1024 == 0, "swizzle atoms");
static_assert(kPrepSmem <= 232448, "shared memory budget");
// TMEM: K'K'^T double-buffered (64 each), W (128), U~ (128), and the A operands
// of the W and U~ MMAs: T diag(beta gamma) hi, lo, T diag(beta) hi, lo (32
// columns each: bf16 pairs (k, k + 1) per column, rows in the M = 64 lanes)
constexpr uint32_t kColKK = 0, kColW = 128, kColU = 256, kColTm = 384, kPrepTmCols = 512;

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

// Arrivals: raw_empty, prep_full one per front-end warp; kk_free, t_ready one
// per inverse warp; t_free, tm_ready, wu_free one per epilogue warp; the rest
// the TMA transaction or one MMA commit.
struct PrepBars {
  uint64_t raw_full[2], raw_empty[2], prep_full[kPrepSlots], prep_empty[kPrepSlots], kk_ready[2], kk_free[2];
  uint64_t tm_ready, tm_free, wu_ready, wu_free, t_ready, t_free;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(PrepBars) <= 256, "barrier block");

// AND of a predicate over the 128 threads of named barrier 1 (the inverse
// warps), so that they leave their loop together
__device__ __forceinline__ bool inv_all(bool ok) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %1, 0;\n\t"
      "bar.red.and.pred p, 1, 128, p;\n\tselp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(r)
      : "r"((uint32_t)ok)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void inv_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
// the 128 threads of the epilogue warps
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 2, 128;" ::: "memory"); }

// kConv, kL2: the front end's convolution and L2 norm as template parameters
// (one code path per instance)
template <bool kConv, bool kL2>
__global__ void __launch_bounds__(kPrepThreads, 1)
    gdn_prep_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv, const PrepParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  PrepBars *bars = reinterpret_cast<PrepBars *>(smem + kOffPBar);
  volatile int *abort = &bars->abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = p.H, T = p.T, nch = p.nchunks;
  const int Cch = 3 * H * kD;
  const int nitems = p.B * H * nch;
  // item w: head fastest, then chunk, then batch
  auto decode = [&](int w, int &b, int &h, int &c) {
    h = w % H;
    const int r = w / H;
    c = r % nch;
    b = r / nch;
  };

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->raw_full[i], 1);
      mbar_init(&bars->raw_empty[i], kFeWarps);
      mbar_init(&bars->kk_ready[i], 1);
      mbar_init(&bars->kk_free[i], 4);
    }
    for (int i = 0; i < kPrepSlots; ++i) {
      mbar_init(&bars->prep_full[i], kFeWarps);
      mbar_init(&bars->prep_empty[i], 1);
    }
    mbar_init(&bars->tm_ready, 4);
    mbar_init(&bars->tm_free, 1);
    mbar_init(&bars->wu_ready, 1);
    mbar_init(&bars->wu_free, 4);
    mbar_init(&bars->t_ready, 4);
    mbar_init(&bars->t_free, 4);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, kPrepTmCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp == 0) {
    // ======================= TMA: raw q, k, v rows =======================
    if (lane == 0) {
      prefetch_tensormap(&tq);
      prefetch_tensormap(&tk);
      prefetch_tensormap(&tv);
      const CUtensorMap *maps[3] = {&tq, &tk, &tv};
      int it = 0;
      for (int w = blockIdx.x; w < nitems; w += gridDim.x, ++it) {
        int b, h, c;
        decode(w, b, h, c);
        const int slot = it & 1;
        if (!wait_bar(&bars->raw_empty[slot], ((uint32_t)(it >> 1) & 1u) ^ 1u, abort)) break;
        uint8_t *raw = smem + kOffRaw + slot * kRawBytes;
        mbar_arrive_expect_tx(&bars->raw_full[slot], kRawBytes);
#pragma unroll
        for (int part = 0; part < 3; ++part)
#pragma unroll
          for (int blk = 0; blk < 2; ++blk)
            tma_load_4d(raw + part * 16384 + blk * 8192, maps[part], &bars->raw_full[slot], 64 * blk, h, c * kC, b);
        // the next item's rows into L2 while this one is in flight
        const int wn = w + gridDim.x;
        if (wn < nitems) {
          int bn, hn, cn;
          decode(wn, bn, hn, cn);
#pragma unroll
          for (int part = 0; part < 3; ++part) {
            tma_prefetch_l2_4d(maps[part], 0, hn, cn * kC, bn);
            tma_prefetch_l2_4d(maps[part], 64, hn, cn * kC, bn);
          }
        }
      }
    }
  } else if (warp == 1) {
    // ======================= MMA issuer =======================
    if (lane == 0) {
      constexpr uint32_t id_kk = idesc_bf16(64, 64, false, false);   // K' K'^T
      constexpr uint32_t id_wu = idesc_bf16(64, 128, false, true);   // Tm K' and Tm V'
      const uint32_t sbase = smem_u32(smem);
      // Two streams of MMAs, issued in whichever order their inputs land:
      // K'K'^T of item ik once its front end is done, W and U~ of item iu once
      // its inverse is done (K'K'^T of item iu + 1 never waits for W, U~ of iu).
      const int nmine = blockIdx.x < (unsigned)nitems ? (nitems - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
      int ik = 0, iu = 0;
      uint64_t t0 = global_timer_ns();
      while (iu < nmine) {
        bool progressed = false;
        if (ik < nmine) {
          const int ps = ik % kPrepSlots, ks2 = ik & 1;
          if (mbar_test(&bars->prep_full[ps], (uint32_t)(ik / kPrepSlots) & 1u) &&
              mbar_test(&bars->kk_free[ks2], ((uint32_t)(ik >> 1) & 1u) ^ 1u)) {
            tc_fence_after();
            // K' K'^T: M = 64, N = 64, K = d_k
            const uint64_t dK = desc_sw128(sbase + kOffPrep + ps * 2 * kPrepTile, 16, 1024);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
              const uint32_t off = ((ks >> 2) * 8192 + (ks & 3) * 32) >> 4;
              umma_bf16(tmem + kColKK + ks2 * 64, dK + off, dK + off, id_kk, ks > 0);
            }
            umma_commit(&bars->kk_ready[ks2]);
            ++ik;
            progressed = true;
          }
        }
        if (iu < ik) {
          const int ps = iu % kPrepSlots;
          const uint32_t pt = (uint32_t)iu & 1u;
          if (mbar_test(&bars->tm_ready, pt) && mbar_test(&bars->wu_free, pt ^ 1u)) {
            tc_fence_after();
            // W = [Tm1_hi | Tm1_lo] K', U~ = [Tm2_hi | Tm2_lo] V': M = 64, N = 128, K = 2 x 64
            // tokens, the A operands in tensor memory (8 columns per 16 tokens)
            const uint64_t dK = desc_sw128(sbase + kOffPrep + ps * 2 * kPrepTile, 8192, 1024);
            const uint64_t dV = desc_sw128(sbase + kOffPrep + ps * 2 * kPrepTile + kPrepTile, 8192, 1024);
#pragma unroll
            for (int part = 0; part < 2; ++part)
#pragma unroll
              for (int ks = 0; ks < 4; ++ks) {
                const uint32_t acol = kColTm + part * 32 + ks * 8, boff = (ks * 2048) >> 4;
                umma_bf16_tmem_a(tmem + kColW, tmem + acol, dK + boff, id_wu, (part | ks) != 0);
                umma_bf16_tmem_a(tmem + kColU, tmem + acol + 64, dV + boff, id_wu, (part | ks) != 0);
              }
            umma_commit(&bars->wu_ready);
            umma_commit(&bars->tm_free);
            umma_commit(&bars->prep_empty[ps]);
            ++iu;
            progressed = true;
          }
        }
        if (progressed) {
          t0 = global_timer_ns();
        } else {
          if (*abort) break;
          if (global_timer_ns() - t0 > kWaitLimitNs) {
            *abort = 1;
            break;
          }
          __nanosleep(32);
        }
      }
    }
  } else if (warp < kInvWarp0) {
    // ======================= front end =======================
    // A task is (part, 8 consecutive tokens) of the chunk: the warp slides the
    // 4-tap window along its tokens, lane l owning channels 4l .. 4l+3, so every
    // access is 8 bytes per lane and the L2 norm is one warp reduction.  The
    // chunk's rows come from the TMA tile; the 3 rows before the chunk (first
    // task of each part only) from global memory, or conv_in before the
    // sequence (zero without it).
    // Warp fw takes the tasks fw + 6k (k = 0..3), all of part fw % 3 (the
    // part's conv taps are loaded once per chunk), row groups fw / 3 + 2k.
    const int fw = warp - kFeWarp0;
    const int part = fw % 3;
    static_assert(kFeWarps % 3 == 0 && 24 % kFeWarps == 0, "a warp's tasks share one part");
    const __nv_bfloat16 *src = part == 0 ? p.q : (part == 1 ? p.k : p.v);
    // channels 4l .. 4l+3: column block l / 16, 16-byte chunk (l % 16) / 2, half l % 2
    const uint32_t cb = (uint32_t)(lane >> 4), ch = (uint32_t)((lane & 15) >> 1), hb = (uint32_t)(lane & 1) * 8;
    // the conv taps of the chunk's head, the 3 rows before the chunk (row group
    // 0 only) and its gates (warp 0 only)
    float4 nwt[4];
    uint2 nhist[3];
    float2 nga = make_float2(1.f, 1.f), ngb = make_float2(0.f, 0.f);
    auto prefetch = [&](int wn) {
      int b, h, c;
      decode(wn, b, h, c);
      const int t0 = c * kC;
#pragma unroll
      for (int c2 = 0; c2 < 4; ++c2)
        nwt[c2] = kConv ? *reinterpret_cast<const float4 *>(p.conv_w + ((size_t)part * H * kD + h * kD + 4 * lane + c2) * 4)
                        : make_float4(0.f, 0.f, 0.f, 1.f);
#pragma unroll
      for (int m = 0; m < 3; ++m) {
        const int t = t0 - 3 + m;
        uint2 v = make_uint2(0u, 0u);
        if (fw < 3) {
          if (t >= 0)
            v = *reinterpret_cast<const uint2 *>(src + (((size_t)b * T + t) * H + h) * kD + 4 * lane);
          else if (kConv && p.conv_in)
            v = *reinterpret_cast<const uint2 *>(p.conv_in + ((size_t)b * 3 + (t + 3)) * Cch + part * H * kD +
                                                 h * kD + 4 * lane);
        }
        nhist[m] = v;
      }
      if (fw == 0) {
        const int ta = t0 + 2 * lane, tb = ta + 1;
        const size_t ia = ((size_t)b * T + ta) * H + h, ib = ((size_t)b * T + tb) * H + h;
        nga = make_float2(ta < T ? p.alpha[ia] : 1.f, tb < T ? p.alpha[ib] : 1.f);
        ngb = make_float2(ta < T ? p.beta[ia] : 0.f, tb < T ? p.beta[ib] : 0.f);
      }
    };
    if (blockIdx.x < (unsigned)nitems) prefetch(blockIdx.x);
    int it = 0;
    for (int w = blockIdx.x; w < nitems; w += gridDim.x, ++it) {
      int b, h, c;
      decode(w, b, h, c);
      const int t0 = c * kC;
      const size_t unit = (size_t)b * H + h;
      const int slot = it & 1, ps = it % kPrepSlots;
      const uint32_t ph = (uint32_t)(it >> 1) & 1u, pph = (uint32_t)(it / kPrepSlots) & 1u;
      // the 4 taps of channels 4l .. 4l+3, as (4l, 4l + 2) and (4l + 1, 4l + 3) pairs
      float4 wt[4];
#pragma unroll
      for (int c2 = 0; c2 < 4; ++c2) wt[c2] = nwt[c2];
      const float2 we[4] = {make_float2(wt[0].x, wt[2].x), make_float2(wt[0].y, wt[2].y), make_float2(wt[0].z, wt[2].z),
                            make_float2(wt[0].w, wt[2].w)};
      const float2 wo[4] = {make_float2(wt[1].x, wt[3].x), make_float2(wt[1].y, wt[3].y), make_float2(wt[1].z, wt[3].z),
                            make_float2(wt[1].w, wt[3].w)};
      // this chunk's history rows and gates were loaded one chunk ahead
      const uint2 hist[3] = {nhist[0], nhist[1], nhist[2]};
      const float a0 = nga.x, a1 = nga.y, be0 = ngb.x, be1 = ngb.y;
      if (w + (int)gridDim.x < nitems) prefetch(w + gridDim.x);
      // W, U~ of chunk it - 3 are done
      if (!wait_bar_warp(&bars->prep_empty[ps], pph ^ 1u, abort)) break;
      if (fw == 0) {
        // gates of the chunk: g2 = cumsum(log2 alpha); alpha = 1, beta = 0 past T
        float *g2s = reinterpret_cast<float *>(smem + kOffPG + ps * 512);
        float *betas = g2s + kC;
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
        betas[2 * lane] = be0;
        betas[2 * lane + 1] = be1;
        p.Gp[unit * p.Tp + t0 + 2 * lane] = ga;
        p.Gp[unit * p.Tp + t0 + 2 * lane + 1] = gb;
      }
      if (!wait_bar_warp(&bars->raw_full[slot], ph, abort)) break;
      const uint8_t *raw = smem + kOffRaw + slot * kRawBytes + part * 16384 + cb * 8192;
      uint8_t *dst_tile = smem + kOffPrep + ps * 2 * kPrepTile + (part == 1 ? 0 : kPrepTile);
#pragma unroll 1
      for (int k = 0; k < 4; ++k) {
        const int r0 = (fw / 3 + 2 * k) * 8;  // the task's 8 tokens
        // channels (4l, 4l + 2) and (4l + 1, 4l + 3) of rows r0 - 3 .. r0 + 7 as
        // fp32 pairs: the even and the odd channels of the lane's 8 bytes
        float2 xe[11], xo[11];
#pragma unroll
        for (int m = 0; m < 11; ++m) {
          const int tr = r0 - 3 + m;
          const uint2 v = tr >= 0 ? *reinterpret_cast<const uint2 *>(raw + swz(tr, ch) + hb) : hist[m < 3 ? m : 0];
          xe[m] = fe::bf16_lows(v.x, v.y);
          xo[m] = fe::bf16_highs(v.x, v.y);
        }
        // the 8 rows are independent: each step runs over all of them
        float2 ye[8], yo[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          ye[r] = fe::conv4x2(we[0], we[1], we[2], we[3], xe[r], xe[r + 1], xe[r + 2], xe[r + 3]);
          yo[r] = fe::conv4x2(wo[0], wo[1], wo[2], wo[3], xo[r], xo[r + 1], xo[r + 2], xo[r + 3]);
        }
        if (part < 2 && kL2) {
          // this lane's ((y0^2 + y1^2) + (y2^2 + y3^2)), then across the lanes
          float ss[8];
#pragma unroll
          for (int r = 0; r < 8; ++r) {
            const float2 pe = __fmul2_rn(ye[r], ye[r]), po = __fmul2_rn(yo[r], yo[r]);
            ss[r] = __fadd_rn(__fadd_rn(pe.x, po.x), __fadd_rn(pe.y, po.y));
          }
          const float inv = fe::inv_norm(fe::warp_pairwise_sum8(ss, lane));
#pragma unroll
          for (int r = 0; r < 8; ++r) {
            const float ir = __shfl_sync(0xffffffffu, inv, fe::row_lane(r));
            const float2 i2 = make_float2(ir, ir);
            ye[r] = __fmul2_rn(ye[r], i2);
            yo[r] = __fmul2_rn(yo[r], i2);
          }
        }
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          const bool valid = t0 + r0 + r < T;
          uint2 pk = make_uint2(0u, 0u);
          if (valid) {
            pk.x = bits(__floats2bfloat162_rn(ye[r].x, yo[r].x));
            pk.y = bits(__floats2bfloat162_rn(ye[r].y, yo[r].y));
          }
          const int t = r0 + r;
          const size_t grow = (unit * p.Tp + t0 + t) * kD + 4 * lane;
          if (part == 0) {
            *reinterpret_cast<uint2 *>(p.Qp + grow) = pk;
          } else {
            *reinterpret_cast<uint2 *>(dst_tile + cb * 8192 + swz(t, ch) + hb) = pk;
            if (part == 1) *reinterpret_cast<uint2 *>(p.Kp + grow) = pk;
          }
        }
      }
      fence_proxy_async_smem();
      warp_arrive(&bars->prep_full[ps]);
      warp_arrive(&bars->raw_empty[slot]);
    }
  } else if (warp < kEpiWarp0) {
    // ======================= A, the inverse and the T tiles =======================
    const int iw = warp - kInvWarp0, itid = tid - 32 * kInvWarp0;  // 0..3, 0..127
    const int q4 = warp & 3;
    const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
    const int r0 = 16 * q4 + (lane >> 2), cq = 2 * (lane & 3);
    float *A00 = reinterpret_cast<float *>(smem + kOffAT);
    float *A10 = A00 + kBlk * kLd;
    float *A11 = A10 + kBlk * kLd;
    float *T00 = A11 + kBlk * kLd;
    float *T10 = T00 + kBlk * kLd;
    float *T11 = T10 + kBlk * kLd;
    int it = 0;
    for (int w = blockIdx.x; w < nitems; w += gridDim.x, ++it) {
      const int slot = it & 1, ps = it % kPrepSlots;
      const uint32_t ph = (uint32_t)(it >> 1) & 1u;
      bool ok = wait_bar_warp(&bars->prep_full[ps], (uint32_t)(it / kPrepSlots) & 1u, abort) &&
                wait_bar_warp(&bars->kk_ready[slot], ph, abort);
      if (!inv_all(ok)) break;
      const float *g2s = reinterpret_cast<const float *>(smem + kOffPG + ps * 512);
      const float *betas = g2s + kC;
      tc_fence_after();
      // ---- A_ij = beta_i 2^(g_i - g_j) (k_i . k_j) for j < i, as the blocks A00, A10, A11
      {
        float kk[32];
        tmem_ld16x256b_x8(tmem + kColKK + slot * 64 + lane_base, kk);
        tc_fence_before();
        warp_arrive(&bars->kk_free[slot]);
        const float gr[2] = {g2s[r0], g2s[r0 + 8]}, br[2] = {betas[r0], betas[r0 + 8]};
#pragma unroll
        for (int m = 0; m < 8; ++m) {  // the pair of columns j, j + 1 of rows r0, r0 + 8
          const int j = 8 * m + cq;
          const float2 gj = *reinterpret_cast<const float2 *>(g2s + j);
#pragma unroll
          for (int rr = 0; rr < 2; ++rr) {
            const int i = r0 + 8 * rr;
            // computed for every (i, j), then selected: no divergent branches
            const float d0 = exp2f(fminf(gr[rr] - gj.x, 0.f)), d1 = exp2f(fminf(gr[rr] - gj.y, 0.f));
            const float a0 = j < i ? br[rr] * d0 * kk[4 * m + 2 * rr] : 0.f;
            const float a1 = j + 1 < i ? br[rr] * d1 * kk[4 * m + 2 * rr + 1] : 0.f;
            // the diagonal blocks transposed (the solve walks their columns), A10 by rows
            if (i < kBlk) {
              if (j < kBlk) {
                A00[j * kLd + i] = a0;
                A00[(j + 1) * kLd + i] = a1;
              }
            } else if (j < kBlk) {
              *reinterpret_cast<float2 *>(A10 + (i - kBlk) * kLd + j) = make_float2(a0, a1);
            } else {
              A11[(j - kBlk) * kLd + (i - kBlk)] = a0;
              A11[(j + 1 - kBlk) * kLd + (i - kBlk)] = a1;
            }
          }
        }
      }
      // the epilogue warps have read T of the previous chunk
      ok = wait_bar_warp(&bars->t_free, ((uint32_t)it & 1u) ^ 1u, abort);
      if (!inv_all(ok)) break;  // also orders the writes of A before the reads below
      // ---- T00 = (I + A00)^-1 (warp 0) and T11 = (I + A11)^-1 (warp 1), each in
      // 16 x 16 sub-blocks [Ta 0; Tb Tc]: the diagonal ones by forward
      // substitution (lanes 0-15 Ta, 16-31 Tc, lane = column c), right-looking:
      // x = e_c, then for i = 0, 1, ...: x_i is final and x_m -= A_mi x_i for
      // m > i (row i of the stored transpose holds column i of A; its entries
      // m <= i are 0 and skipped); then Tb = -Tc (Ab Ta).
      if (iw < 2) {
        const float *At = iw ? A11 : A00;
        float *Tb = iw ? T11 : T00;
        const int hf = lane >> 4, c = lane & 15, base = 16 * hf;
        float x[16];
#pragma unroll
        for (int m = 0; m < 16; ++m) x[m] = m == c ? 1.f : 0.f;
#pragma unroll
        for (int i = 0; i < 15; ++i) {
#pragma unroll
          for (int m4 = ((i + 1) / 4) * 4; m4 < 16; m4 += 4) {
            const float4 a = *reinterpret_cast<const float4 *>(At + (base + i) * kLd + base + m4);
            const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if (m4 + e > i) x[m4 + e] = fmaf(-av[e], x[i], x[m4 + e]);
          }
        }
        // Ta, Tc by rows, and the zero block above Tc
#pragma unroll
        for (int m = 0; m < 16; ++m) {
          Tb[(base + m) * kLd + base + c] = x[m];
          if (hf) Tb[m * kLd + 16 + c] = 0.f;
        }
        // P = Ab Ta (Ab = A[16..31][0..15], i.e. rows 0-15, columns 16-31 of the
        // transpose): column c, rows 8 hf .. 8 hf + 7 in this lane
        float ta[16];
#pragma unroll
        for (int m = 0; m < 16; ++m) ta[m] = __shfl_sync(0xffffffffu, x[m], c);
        float pr[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) pr[r] = 0.f;
#pragma unroll
        for (int m = 0; m < 16; ++m) {
          const float4 u = *reinterpret_cast<const float4 *>(At + m * kLd + 16 + 8 * hf);
          const float4 v = *reinterpret_cast<const float4 *>(At + m * kLd + 20 + 8 * hf);
          pr[0] = fmaf(u.x, ta[m], pr[0]); pr[1] = fmaf(u.y, ta[m], pr[1]);
          pr[2] = fmaf(u.z, ta[m], pr[2]); pr[3] = fmaf(u.w, ta[m], pr[3]);
          pr[4] = fmaf(v.x, ta[m], pr[4]); pr[5] = fmaf(v.y, ta[m], pr[5]);
          pr[6] = fmaf(v.z, ta[m], pr[6]); pr[7] = fmaf(v.w, ta[m], pr[7]);
        }
        float pc[16];  // column c of P
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          const float o = __shfl_xor_sync(0xffffffffu, pr[r], 16);
          pc[r] = hf ? o : pr[r];
          pc[8 + r] = hf ? pr[r] : o;
        }
        __syncwarp();  // Tc's rows are stored
        // Tb = -Tc P: rows 8 hf .. 8 hf + 7 of column c
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          const float *tc = Tb + (16 + 8 * hf + r) * kLd + 16;
          float acc = 0.f;
#pragma unroll
          for (int m4 = 0; m4 < 16; m4 += 4) {
            const float4 t4 = *reinterpret_cast<const float4 *>(tc + m4);
            acc = fmaf(t4.x, pc[m4], acc);
            acc = fmaf(t4.y, pc[m4 + 1], acc);
            acc = fmaf(t4.z, pc[m4 + 2], acc);
            acc = fmaf(t4.w, pc[m4 + 3], acc);
          }
          Tb[(16 + 8 * hf + r) * kLd + c] = -acc;
        }
      }
      inv_sync();
      // ---- T10 = -T11 (A10 T00): X = A10 T00 in A00's place, then T10 = -T11 X;
      // thread: row itid >> 2, columns 8 (itid & 3) .. + 7
      float *X = A00;
      {
        const int r = itid >> 2, c0 = 8 * (itid & 3);
        // acc[0..7] += sum_m L[r][m] R[m][c0 .. c0 + 7], rows of 16-byte groups
        auto rowprod = [&](const float *L, const float *R, float (&acc)[8]) {
#pragma unroll
          for (int q = 0; q < 8; ++q) acc[q] = 0.f;
#pragma unroll
          for (int m4 = 0; m4 < kBlk; m4 += 4) {
            const float4 l = *reinterpret_cast<const float4 *>(L + r * kLd + m4);
            const float lv[4] = {l.x, l.y, l.z, l.w};
#pragma unroll
            for (int mm = 0; mm < 4; ++mm) {
              const float4 ra = *reinterpret_cast<const float4 *>(R + (m4 + mm) * kLd + c0);
              const float4 rb = *reinterpret_cast<const float4 *>(R + (m4 + mm) * kLd + c0 + 4);
              acc[0] = fmaf(lv[mm], ra.x, acc[0]); acc[1] = fmaf(lv[mm], ra.y, acc[1]);
              acc[2] = fmaf(lv[mm], ra.z, acc[2]); acc[3] = fmaf(lv[mm], ra.w, acc[3]);
              acc[4] = fmaf(lv[mm], rb.x, acc[4]); acc[5] = fmaf(lv[mm], rb.y, acc[5]);
              acc[6] = fmaf(lv[mm], rb.z, acc[6]); acc[7] = fmaf(lv[mm], rb.w, acc[7]);
            }
          }
        };
        float acc[8];
        rowprod(A10, T00, acc);
        *reinterpret_cast<float4 *>(X + r * kLd + c0) = make_float4(acc[0], acc[1], acc[2], acc[3]);
        *reinterpret_cast<float4 *>(X + r * kLd + c0 + 4) = make_float4(acc[4], acc[5], acc[6], acc[7]);
        inv_sync();
        rowprod(T11, X, acc);
        *reinterpret_cast<float4 *>(T10 + r * kLd + c0) = make_float4(-acc[0], -acc[1], -acc[2], -acc[3]);
        *reinterpret_cast<float4 *>(T10 + r * kLd + c0 + 4) = make_float4(-acc[4], -acc[5], -acc[6], -acc[7]);
      }
      warp_arrive(&bars->t_ready);
      inv_sync();  // the next chunk's A may overwrite the blocks read above
    }
  } else {
    // ============ the T tiles, then W (bf16) and U~ (fp32) to global memory ============
    const int etid = tid - 32 * kEpiWarp0;  // 0..127
    const float *T00 = reinterpret_cast<const float *>(smem + kOffAT) + 3 * kBlk * kLd;
    const float *T10 = T00 + kBlk * kLd;
    const float *T11 = T10 + kBlk * kLd;
    const int q4 = warp & 3;
    const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
    const int r0 = 16 * q4 + (lane >> 2), cq = 2 * (lane & 3);
    int it = 0;
    for (int w = blockIdx.x; w < nitems; w += gridDim.x, ++it) {
      int b, h, c;
      decode(w, b, h, c);
      const size_t unit = (size_t)b * H + h;
      const size_t row0 = unit * p.Tp + c * kC + r0, row1 = row0 + 8;
      const int slot = it & 1;
      // ---- T diag(beta gamma) and T diag(beta) as bf16 hi / lo MMA operands in
      // tensor memory, once the inverse is done and the previous chunk's W and U~
      // MMAs have read them
      if (!wait_bar_warp(&bars->t_ready, (uint32_t)it & 1u, abort)) break;
      if (!wait_bar_warp(&bars->tm_free, ((uint32_t)it & 1u) ^ 1u, abort)) break;
      float *colbg = reinterpret_cast<float *>(smem + kOffCol) + slot * 2 * kC;
      float *colb = colbg + kC;
      if (etid < kC) {
        const float *g2s = reinterpret_cast<const float *>(smem + kOffPG + (it % kPrepSlots) * 512);
        const float bk = g2s[kC + etid];
        colbg[etid] = bk * exp2f(g2s[etid]);
        colb[etid] = bk;
      }
      epi_sync();
      tc_fence_after();
      {
        // 16x256b fragment: rows r0, r0 + 8; column pairs k = 16m + 4(lane & 3) .. + 3
        // (T01 = 0; T00, T10 or T11 otherwise)
        const int q = lane & 3;
        float tv[2][4][4];
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
          const int i = r0 + 8 * rr;
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const int k = 16 * m + 4 * q;
            const float *src = i < kBlk ? (k < kBlk ? T00 + i * kLd + k : nullptr)
                                        : (k < kBlk ? T10 + (i - kBlk) * kLd + k : T11 + (i - kBlk) * kLd + (k - kBlk));
            const float4 t4 = src ? *reinterpret_cast<const float4 *>(src) : make_float4(0.f, 0.f, 0.f, 0.f);
            tv[rr][m][0] = t4.x; tv[rr][m][1] = t4.y; tv[rr][m][2] = t4.z; tv[rr][m][3] = t4.w;
          }
        }
#pragma unroll
        for (int part = 0; part < 2; ++part) {  // T diag(beta gamma), T diag(beta)
          const float *col = part ? colb : colbg;
          uint32_t vh[16], vl[16];
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const float4 cs = *reinterpret_cast<const float4 *>(col + 16 * m + 4 * q);
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
              split2(tv[rr][m][0] * cs.x, tv[rr][m][1] * cs.y, vh[4 * m + 2 * rr], vl[4 * m + 2 * rr]);
              split2(tv[rr][m][2] * cs.z, tv[rr][m][3] * cs.w, vh[4 * m + 2 * rr + 1], vl[4 * m + 2 * rr + 1]);
            }
          }
          tmem_st16x256b_x4(tmem + kColTm + part * 64 + lane_base, vh);
          tmem_st16x256b_x4(tmem + kColTm + part * 64 + 32 + lane_base, vl);
        }
        tmem_wait_st();
      }
      tc_fence_before();
      warp_arrive(&bars->tm_ready);
      warp_arrive(&bars->t_free);
      if (!wait_bar_warp(&bars->wu_ready, (uint32_t)it & 1u, abort)) break;
      tc_fence_after();
      float v0[32], v1[32];
      tmem_ld16x256b_x8x2(tmem + kColW + lane_base, tmem + kColW + 64 + lane_base, v0, v1);
#pragma unroll
      for (int m = 0; m < 16; ++m) {
        const float *v = m < 8 ? v0 : v1;
        const int mm = m & 7, col = 8 * m + cq;
        *reinterpret_cast<__nv_bfloat162 *>(p.Wp + row0 * kD + col) = __floats2bfloat162_rn(v[4 * mm], v[4 * mm + 1]);
        *reinterpret_cast<__nv_bfloat162 *>(p.Wp + row1 * kD + col) =
            __floats2bfloat162_rn(v[4 * mm + 2], v[4 * mm + 3]);
      }
      tmem_ld16x256b_x8x2(tmem + kColU + lane_base, tmem + kColU + 64 + lane_base, v0, v1);
      tc_fence_before();
      warp_arrive(&bars->wu_free);
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
  if (*abort && tid == 0 && p.dev_status) atomicOr(p.dev_status, GLINATTN_DEV_WAIT_TIMEOUT);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kPrepTmCols);
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
    const int bad = gates_bad(p.alpha + (size_t)b * T * p.H + h, T, p.H, tid, kThreads);
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
        if (!wait_bar<false>(&bars->empty[s], ((uint32_t)(c / kStages) & 1u) ^ 1u, abort)) break;
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
        if (!wait_bar<false>(&bars->full[s], (uint32_t)(c / kStages) & 1u, abort)) break;
        if (!wait_bar<false>(&bars->s_ready, pc, abort)) break;
        tc_fence_after();
        // W [S_hi | S_lo]: M = 64, N = 64, K = d_k (W tile K-major, S tile MN-major)
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t aoff = ((ks >> 2) * (kTile / 2) + (ks & 3) * 32) >> 4;
          umma_bf16(tmem + kColWS, dW + aoff, dS + ((ks * 2048) >> 4), id_xs, ks > 0);
        }
        umma_commit(&bars->ws_ready);
        if (!wait_bar<false>(&bars->u_ready, pc, abort)) break;
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
      if (!wait_bar_warp<false>(&bars->qk_ready, pc, abort)) break;
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
      if (!wait_bar_warp<false>(&bars->p_free, pc ^ 1u, abort)) break;
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
      if (!wait_bar_warp<false>(&bars->ws_ready, pc, abort)) { ok = false; break; }
      tc_fence_after();
      float ws[32];
      tmem_ld16x256b_x8(tmem + kColWS + lane_base, ws);
      if (!wait_bar_warp<false>(&bars->full[s], sph, abort)) { ok = false; break; }
      if (!wait_bar_warp<false>(&bars->p_free, pc ^ 1u, abort)) { ok = false; break; }
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
      if (!wait_bar_warp<false>(&bars->ds_ready, pc, abort)) { ok = false; break; }
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
      if (!wait_bar_warp<false>(&bars->o_ready, pc, abort)) { ok = false; break; }
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
        if (!wait_bar<false>(&bars->ws_ready, pc, abort)) break;
        if (!wait_bar<false>(&bars->o_free, pc ^ 1u, abort)) break;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t aoff = ((ks >> 2) * (kTile / 2) + (ks & 3) * 32) >> 4;
          umma_bf16(tmem + kColO, dQ + aoff, dS + ((ks * 2048) >> 4), id_xs, ks > 0);
        }
        // (P''hi + P''lo) [U_hi | U_lo] into the same columns, once K'^T r U is done
        if (!wait_bar<false>(&bars->ds_ready, pc, abort)) break;
        if (!wait_bar<false>(&bars->p_ready, pc, abort)) break;
        if (!wait_bar<false>(&bars->u_ready, pc, abort)) break;
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
        if (!wait_bar<false>(&bars->full[s], (uint32_t)(c / kStages) & 1u, abort)) break;
        if (!wait_bar<false>(&bars->qk_free, ((uint32_t)c & 1u) ^ 1u, abort)) break;
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
  // persistent: one CTA per SM (or per item when there are fewer)
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return GLINATTN_ERR_CUDA;
  const long long items = (long long)B * H * nchunks;
  const unsigned grid = (unsigned)(items < sms ? items : sms);
  prep<<<grid, kPrepThreads, kPrepSmem, stream>>>(rq, rk, rv, pp);
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
