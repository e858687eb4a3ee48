// prefill_tc.cu -- chunked prefill on the 5th-generation tensor cores.
//
// "Inference for linear attention and hybrid architectures", section "Two
// ways to write the same computation": prefill splits the sequence into chunks
// of C tokens; inside a chunk the work is a C x C decay-masked "attention"
// done with matrix multiplies, and only the d_k x d_v state passes from one
// chunk to the next.  With g the cumulative log decay inside the chunk,
// gamma = exp(g), D_ij = exp(g_i - g_j) [j <= i] and r_j = exp(g_C - g_j):
//
//   O      = diag(gamma) Q S + ((Q K^T) * D) V
//   S_next = gamma_C S + K^T diag(r) V
//
// (the page's chunked gated linear attention; the decay of the state update
// is applied to V's rows here instead of K's, which is the same product).
//
// Kernel design (sm_103a):
//   * one CTA per (batch, head, 64-wide slice of d_v: two slices at d_v = 128,
//     one in the SSD form's d_v = 64); groups of heads may share q and k
//     (the q / k tiles come from head h / (H / Hq)); the state slice
//     S[128 x 64] is fp32 and lives in the registers of the epilogue warps
//     for the whole sequence, one d_k row per thread of warpgroup B;
//   * warp 0 streams Q, K (64 x 128) and V (64 x 64) chunk tiles with TMA
//     (128-byte swizzle, 3-stage ring, out-of-range rows of a ragged last
//     chunk are zero-filled by the copy engine) and the chunk's gates into a
//     ring beside them, prefetching 3 more chunks into L2;
//   * two threads issue tcgen05.mma (a thread issues one small MMA about every
//     85 cycles, so the chunk's MMAs are spread over two issuers): warp 1 the
//     state chain, K^T V~ and then Q S; warp 10 Q K^T one chunk ahead and P V.
//     Accumulators in TMEM: Q K^T and P V double-buffered (64 columns each),
//     Q [S_hi | S_lo] and K^T [V~hi | V~lo] (128 columns each);
//   * warpgroup A (warps 2-5) forms P = (QK^T)*D and V~ = diag(r) V as bf16
//     hi / lo tiles; warpgroup B (warps 6-9) holds the state, folds the
//     K^T V~ accumulator into it, writes the next state's hi / lo tile and
//     writes the outputs gamma_i (Q S)_i + (P V)_i.  Operands derived in fp32
//     (P, V~, S) are split into a bf16 high part and a bf16 remainder and
//     multiplied twice, so the products keep ~16 bits instead of bf16's 8 (one
//     bf16 rounding of these operands alone costs ~2e-3 relative error in o
//     and S).
//   Every mbarrier wait is bounded; on timeout the CTA raises
//   GLINATTN_DEV_WAIT_TIMEOUT and all roles leave their loops.
#include <cuda.h>
#include <cuda_bf16.h>
#include <stdio.h>
#include <string.h>

#include "common.cuh"
#include "prefill_tc.cuh"
#include "sm100.cuh"
#include "tc_common.cuh"

namespace glinattn {
namespace {

using namespace sm100;
using namespace tc;

constexpr int kC = 64;    // chunk length
constexpr int kDK = 128;  // key / value head size
constexpr int kBV = 64;   // d_v columns per CTA
constexpr int kStages = 3;
constexpr int kPrefetch = 3;  // chunks prefetched into L2 beyond the shared-memory ring
// warp 0 TMA and gates, warp 1 MMA issuer of the state chain (K^T V~, Q S),
// warps 2-5 and 6-9 epilogue, warp 10 MMA issuer of Q K^T and P V
constexpr int kThreads = 352;
constexpr int kEpiThreads = 128;  // threads per epilogue warpgroup

// ---- shared memory map (offsets from a 1024-byte aligned base) -------------
constexpr uint32_t kTileQ = kC * kDK * 2;  // 16 KiB: two 64-column swizzled blocks
constexpr uint32_t kTileK = kC * kDK * 2;  // 16 KiB
constexpr uint32_t kTileV = kC * kBV * 2;  // 8 KiB
constexpr uint32_t kStageBytes = kTileQ + kTileK + kTileV;
constexpr uint32_t kTileP = kC * kC * 2;   // 8 KiB, one of hi / lo
constexpr uint32_t kTileS = kDK * kBV * 2; // 16 KiB, one of hi / lo
constexpr uint32_t kOffStage = 0;
constexpr uint32_t kOffP = kOffStage + kStages * kStageBytes;  // P[hi, lo]
constexpr uint32_t kOffVt = kOffP + 2 * kTileP;                // V~[hi, lo]
constexpr uint32_t kOffS = kOffVt + 2 * kTileV;                // S[buf][hi, lo]
constexpr uint32_t kOffG = kOffS + 4 * kTileS;                 // gate ring [stage]
constexpr uint32_t kGateBytes = 1088;                          // one GateRing entry
constexpr uint32_t kOffBar = kOffG + kStages * kGateBytes;
constexpr uint32_t kSmemBytes = kOffBar + 256 + 1024;  // barriers + alignment slack
// the normalised variant only, past the barriers: 1 / denominator ring
// [slot][token], the chunk's column sums of phi(k) [stage][d_k] and z at the
// chunk start, one copy per warp of warpgroup A [4][d_k]
constexpr int kDenSlots = 4;
constexpr uint32_t kOffDen = kOffBar + 256;
constexpr uint32_t kOffZ = kOffDen + kDenSlots * kC * 4;
constexpr uint32_t kZBytes = kDK * 4;
constexpr uint32_t kOffZrun = kOffZ + kStages * kZBytes;
constexpr uint32_t kSmemBytesNla = kOffZrun + 4 * kZBytes + 1024;
static_assert(kSmemBytesNla <= 232448, "shared memory budget");

// TMEM columns: QK^T double-buffered (64 each), Q[S_hi|S_lo] (128), P V
// double-buffered (64 each), K^T[V~hi|V~lo] (128).
constexpr uint32_t kTmCols = 512;
constexpr uint32_t kColQK = 0, kColO1 = 128, kColO2 = 256, kColDS = 384;

struct GlaParams {
  int B, T, H, nchunks, out_bf16;
  int rep;   // heads per q / k head
  int DV;    // value head size: 128 (two CTAs per head) or 64 (one)
  const int *skip;  // [B, H] or NULL: units to skip (a gate elsewhere in a split sequence is invalid)
  int state_every, nblocks;  // states emitted after every state_every tokens (a multiple of 64)
  float *S_blocks;
  // normalised linear attention (the kNla instances only): the column sums
  // of phi(k) of every chunk [B, Hq, nchunks, d_k], the start normaliser
  // [B, H, d_k] and z_T [B, H, d_k] (NULL: not written); the outputs are
  // divided by phi(q_t) . z_t + 1e-6
  const float *nla_dz;
  const float *nla_z0;
  float *nla_zT;
  const float *alpha;
  const float *S0;
  float *S_T;
  void *o;
  uint32_t *dev_status;
};

struct Bars {
  uint64_t full[kStages], empty[kStages];
  uint64_t qk_ready[2], qk_free[2], p_ready[2], p_free;
  uint64_t ds_ready, ds_free, o_ready[2], o_free[2], s_ready[2];
  uint64_t den_ready[kDenSlots];
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(Bars) <= 256, "barrier block");

// The gates of one chunk, computed once by the TMA warp and published with
// the chunk's tiles: g = cumsum(log2 alpha) over the chunk's tokens (alpha = 1
// past the end of the sequence), 2^g, 2^-g (when the chunk's total decay g_C
// is moderate, so the factors cannot overflow), r = 2^(g_C - g) and 2^g_C.
struct __align__(16) GateRing {
  float g[kC], eg[kC], ecg[kC], r[kC];
  float gC, egC;
  int factored;
};
static_assert(sizeof(GateRing) <= kGateBytes, "gate ring entry");

// kOutBf16, kEmit: the output dtype and whether block states are emitted are
// template parameters, so that each instance carries only its own paths in
// the epilogue loop (a compact loop measured faster than runtime branches).
// kNla: normalised linear attention (gates 1, q and k already the features):
// warpgroup A also carries z from chunk to chunk (each warp its own copy, plus
// the chunk's column sums of phi(k), which arrive with the tiles) and forms
// each token's denominator phi(q_t) . z_t from z at the chunk start and the
// row sum of the masked phi(Q) phi(K)^T; warpgroup B divides the outputs by
// it.  This instance multiplies by no gate and uses two-lane arithmetic in
// its state fold and outputs (faster here, slower in the gated instances).
template <bool kOutBf16, bool kEmit, bool kNla>
__global__ void __launch_bounds__(kThreads, 1)
    gla_prefill_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                       const __grid_constant__ CUtensorMap tv, const GlaParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);  // stays in the shared space
  Bars *bars = reinterpret_cast<Bars *>(smem + kOffBar);
  GateRing *ring = reinterpret_cast<GateRing *>(smem + kOffG);
  volatile int *abort = &bars->abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nvb = p.DV / kBV;
  const int vblk = blockIdx.x % nvb;
  const int bh = blockIdx.x / nvb;
  const int b = bh / p.H, h = bh - b * p.H;
  const int hq = h / p.rep;  // the q / k head of head h
  const int T = p.T, nchunks = p.nchunks;

  // ---- the unit is skipped when a gate is outside (0, 1] ---------------------
  {
    const int bad = p.alpha ? gates_bad(p.alpha + (size_t)b * T * p.H + h, T, p.H, tid, kThreads) : 0;  // no gates: 1
    if (__syncthreads_or(bad)) {
      if (tid == 0 && p.dev_status) atomicOr(p.dev_status, GLINATTN_DEV_BAD_GATE);
      return;
    }
    if (p.skip && p.skip[bh]) {  // uniform over the CTA
      return;
    }
  }

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->full[s], 1 + 32);  // the TMA transaction and the 32 gate lanes
      mbar_init(&bars->empty[s], 2);  // one commit from each MMA issuer
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->qk_ready[i], 1);
      mbar_init(&bars->o_ready[i], 2);  // Q S (issuer A) and P V (issuer B)
      mbar_init(&bars->qk_free[i], kEpiThreads);
      mbar_init(&bars->p_ready[i], kEpiThreads);
      mbar_init(&bars->o_free[i], kEpiThreads);
      mbar_init(&bars->s_ready[i], kEpiThreads);
    }
    for (int i = 0; i < kDenSlots; ++i) mbar_init(&bars->den_ready[i], kEpiThreads);
    mbar_init(&bars->p_free, 2);
    mbar_init(&bars->ds_ready, 1);
    mbar_init(&bars->ds_free, kEpiThreads);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, kTmCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp == 0) {
    // ============ TMA producer (lane 0) and the gates of each chunk (all lanes) ============
    auto prefetch = [&](int c) {  // chunk c's tiles into L2, ahead of the ring
      if (c >= nchunks) return;
      const int t0 = c * kC;
      tma_prefetch_l2_4d(&tq, 0, hq, t0, b);
      tma_prefetch_l2_4d(&tq, 64, hq, t0, b);
      tma_prefetch_l2_4d(&tk, 0, hq, t0, b);
      tma_prefetch_l2_4d(&tk, 64, hq, t0, b);
      tma_prefetch_l2_4d(&tv, vblk * kBV, h, t0, b);
    };
    if (lane == 0) {
      prefetch_tensormap(&tq);
      prefetch_tensormap(&tk);
      prefetch_tensormap(&tv);
      for (int c = 0; c < kPrefetch; ++c) prefetch(kStages + c);
    }
    // lane l holds the alphas of tokens 2l and 2l + 1 of the next chunk
    auto alphas = [&](int c, float &a0, float &a1) {
      const int ta = c * kC + 2 * lane, tb2 = ta + 1;
      a0 = ta < T && p.alpha ? p.alpha[((size_t)b * T + ta) * p.H + h] : 1.f;
      a1 = tb2 < T && p.alpha ? p.alpha[((size_t)b * T + tb2) * p.H + h] : 1.f;
    };
    float a0n, a1n;
    alphas(0, a0n, a1n);
    for (int c = 0; c < nchunks; ++c) {
      const int s = c % kStages;
      const uint32_t use = (uint32_t)(c / kStages);
      if (lane == 0) prefetch(c + kStages + kPrefetch);
      if (!wait_bar_warp<!kNla>(&bars->empty[s], (use & 1u) ^ 1u, abort)) break;
      if (lane == 0) {
        uint8_t *st = smem + kOffStage + s * kStageBytes;
        mbar_arrive_expect_tx(&bars->full[s], kNla ? kStageBytes + kZBytes : kStageBytes);
        const int t0 = c * kC;
        if (kNla)  // the chunk's column sums of phi(k) travel with its tiles
          bulk_load(smem + kOffZ + s * kZBytes, p.nla_dz + (((size_t)b * (p.H / p.rep) + hq) * nchunks + c) * kDK,
                    kZBytes, &bars->full[s]);
        tma_load_4d(st, &tq, &bars->full[s], 0, hq, t0, b);
        tma_load_4d(st + kTileQ / 2, &tq, &bars->full[s], 64, hq, t0, b);
        tma_load_4d(st + kTileQ, &tk, &bars->full[s], 0, hq, t0, b);
        tma_load_4d(st + kTileQ + kTileK / 2, &tk, &bars->full[s], 64, hq, t0, b);
        tma_load_4d(st + kTileQ + kTileK, &tv, &bars->full[s], vblk * kBV, h, t0, b);
      }
      const float l0 = log2f(a0n), l1 = log2f(a1n);
      alphas(c + 1, a0n, a1n);
      float incl = l0 + l1;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      float excl = __shfl_up_sync(0xffffffffu, incl, 1);
      if (lane == 0) excl = 0.f;
      const float ga = excl + l0, gb = excl + l0 + l1;
      const float gC = __shfl_sync(0xffffffffu, gb, 31);
      const bool factored = gC > -100.f;  // 2^-g <= 2^100: no overflow
      GateRing &gr = ring[s];
      gr.g[2 * lane] = ga;
      gr.g[2 * lane + 1] = gb;
      gr.eg[2 * lane] = exp2f(ga);
      gr.eg[2 * lane + 1] = exp2f(gb);
      gr.ecg[2 * lane] = factored ? exp2f(-ga) : 0.f;
      gr.ecg[2 * lane + 1] = factored ? exp2f(-gb) : 0.f;
      gr.r[2 * lane] = exp2f(gC - ga);
      gr.r[2 * lane + 1] = exp2f(gC - gb);
      if (lane == 0) {
        gr.gC = gC;
        gr.egC = exp2f(gC);
        gr.factored = factored ? 1 : 0;
      }
      mbar_arrive(&bars->full[s]);  // releases this lane's gate writes
    }
  } else if (warp == 1) {
    // ============ MMA issuer A: the state chain, K^T V~ and Q S ============
    if (lane == 0) {
      constexpr uint32_t id_qs = idesc_bf16(64, 2 * kBV, false, true);  // Q [S_hi | S_lo]
      constexpr uint32_t id_ds = idesc_bf16(128, 2 * kBV, true, true);  // K^T [V~hi | V~lo]
      const uint32_t sbase = smem_u32(smem);
      const uint64_t dVt = desc_sw128(sbase + kOffVt, kTileV, 1024);  // [hi | lo] as N = 128
      for (int c = 0; c < nchunks; ++c) {
        const int s = c % kStages;
        const int tb = c & 1;
        const uint32_t ph = (uint32_t)(c >> 1) & 1u;
        if (!wait_bar<!kNla>(&bars->p_ready[tb], ph, abort)) break;  // V~ of chunk c
        if (!wait_bar<!kNla>(&bars->ds_free, ((uint32_t)c & 1u) ^ 1u, abort)) break;
        tc_fence_after();
        const uint32_t aQ = sbase + kOffStage + s * kStageBytes;
        const uint32_t aK = aQ + kTileQ;
        // descriptors built once; the k-steps only move the start-address field
        const uint64_t dKm = desc_sw128(aK, kTileK / 2, 1024);
        const uint64_t dQ = desc_sw128(aQ, 16, 1024);
        // dS = K^T [V~hi | V~lo]: M = d_k (K tile read M-major), N = 128, K = 64 tokens
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          umma_bf16(tmem + kColDS, dKm + ((ks * 2048) >> 4), dVt + ((ks * 2048) >> 4), id_ds, ks > 0);
        umma_commit(&bars->ds_ready);
        umma_commit(&bars->p_free);  // V~ may be rewritten
        const int sb = c & 1;
        if (!wait_bar<!kNla>(&bars->s_ready[sb], ph, abort)) break;
        // Q S accumulator is single: the previous chunk's outputs must be read
        if (c > 0 && !wait_bar<!kNla>(&bars->o_free[(c - 1) & 1], (uint32_t)((c - 1) >> 1) & 1u, abort)) break;
        tc_fence_after();
        const uint64_t dS = desc_sw128(sbase + kOffS + sb * 2 * kTileS, kTileS, 1024);  // [hi | lo]
        // O1 = Q [S_hi | S_lo]: M = 64, N = 128, K = d_k (S tile rows = d_k, MN-major)
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t qoff = ((ks >> 2) * (kTileQ / 2) + (ks & 3) * 32) >> 4;
          umma_bf16(tmem + kColO1, dQ + qoff, dS + ((ks * 2048) >> 4), id_qs, ks > 0);
        }
        umma_commit(&bars->o_ready[tb]);
        umma_commit(&bars->empty[s]);
      }
    }
  } else if (warp < 6) {
    // ============ warpgroup A: P = (Q K^T) * D and V~ = diag(r) V ============
    const int q4 = warp & 3;
    const int e = tid - 64;               // 0..127
    const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
    // normalised instance: every warp carries z at the chunk start (lane l
    // channels 4l .. 4l+3) and keeps a copy in shared memory for the
    // denominators of its rows, so no other warp waits on it
    float4 zl = make_float4(0.f, 0.f, 0.f, 0.f);
    float4 *zw = reinterpret_cast<float4 *>(smem + kOffZrun + q4 * kZBytes);
    if (kNla) {
      zl = reinterpret_cast<const float4 *>(p.nla_z0 + ((size_t)b * p.H + h) * kDK)[lane];
      zw[lane] = zl;
      __syncwarp();
    }
    for (int c = 0; c < nchunks; ++c) {
      const int s = c % kStages;
      const uint32_t sph = (uint32_t)(c / kStages) & 1u;
      const int tb = c & 1;
      const uint32_t ph = (uint32_t)(c >> 1) & 1u;
      if (!wait_bar_warp<!kNla>(&bars->qk_ready[tb], ph, abort)) break;
      if (!wait_bar_warp<!kNla>(&bars->full[s], sph, abort)) break;  // the chunk's gates and V tile
      const GateRing &gr = ring[s];
      tc_fence_after();
      // lane l < 16 holds row 16*q4 + l of QK^T (M = 64 layout); it keeps
      // columns 0..31 and hands columns 32..63 to lane l + 16
      float qk[32];
      {
        float lo32[32], hi32[32];
        tmem_ld32x2(tmem + kColQK + tb * 64 + lane_base, tmem + kColQK + tb * 64 + 32 + lane_base, lo32, hi32);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float x = __shfl_sync(0xffffffffu, hi32[j], lane & 15);
          qk[j] = lane < 16 ? lo32[j] : x;
        }
      }
      tc_fence_before();
      mbar_arrive(&bars->qk_free[tb]);
      if (!wait_bar_warp<!kNla>(&bars->p_free, ((uint32_t)c & 1u) ^ 1u, abort)) break;
      // D_ij = 2^(g_i - g_j).  When the chunk's total decay is moderate the
      // factors 2^g_i and 2^-g_j cannot overflow and D is their product (one
      // exp2 per token, done by the TMA warp); otherwise pairwise exp2.
      {
        const int row = 16 * q4 + (lane & 15), jb = 32 * (lane >> 4);
        const uint32_t phi = smem_u32(smem + kOffP);
        const uint32_t plo = phi + kTileP;
        if constexpr (kNla) {  // every gate is 1: D is the causal mask
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) qk[jj] = (jb + jj <= row) ? qk[jj] : 0.f;
        } else if (gr.factored) {  // warp-uniform
          const float rf = gr.eg[row];
          const uint32_t cfa = smem_u32(&gr.ecg[jb]);
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const uint4 cw = lds128(cfa + 16 * q);
            const float cf[4] = {__uint_as_float(cw.x), __uint_as_float(cw.y), __uint_as_float(cw.z),
                                 __uint_as_float(cw.w)};
#pragma unroll
            for (int m = 0; m < 4; ++m) {
              const int jj = 4 * q + m, j = jb + jj;
              qk[jj] = (j <= row) ? qk[jj] * rf * cf[m] : 0.f;
            }
          }
        } else {
          const float gi = gr.g[row];
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) {
            const int j = jb + jj;
            qk[jj] = (j <= row) ? qk[jj] * exp2f(gi - gr.g[j]) : 0.f;
          }
        }
        if (kNla) {
          // phi(q_row) . z over this lane's 64 channels (its half of the Q
          // tile), plus its half of the masked row of phi(Q) phi(K)^T
          const int half = lane >> 4;
          const uint32_t qrow = smem_u32(smem + kOffStage + s * kStageBytes) + half * (kTileQ / 2);
          const float4 *zh = zw + 16 * half;
          // four two-lane partial sums, so the chain of additions stays short
          float2 e[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
          for (int jj = 0; jj < 32; jj += 8) {
#pragma unroll
            for (int m = 0; m < 4; ++m) e[m] = __fadd2_rn(e[m], make_float2(qk[jj + 2 * m], qk[jj + 2 * m + 1]));
          }
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) {
            float x[8];
            unpack8(lds128(qrow + swz(row, ch)), x);
            const float4 za = zh[2 * ch], zb = zh[2 * ch + 1];
            e[0] = __ffma2_rn(make_float2(x[0], x[1]), make_float2(za.x, za.y), e[0]);
            e[1] = __ffma2_rn(make_float2(x[2], x[3]), make_float2(za.z, za.w), e[1]);
            e[2] = __ffma2_rn(make_float2(x[4], x[5]), make_float2(zb.x, zb.y), e[2]);
            e[3] = __ffma2_rn(make_float2(x[6], x[7]), make_float2(zb.z, zb.w), e[3]);
          }
          float den = ((e[0].x + e[0].y) + (e[1].x + e[1].y)) + ((e[2].x + e[2].y) + (e[3].x + e[3].y));
          den += __shfl_xor_sync(0xffffffffu, den, 16);
          if (lane < 16) reinterpret_cast<float *>(smem + kOffDen)[(c & (kDenSlots - 1)) * kC + row] = 1.f / (den + 1e-6f);
          mbar_arrive(&bars->den_ready[c & (kDenSlots - 1)]);
          // z at the next chunk start: plus the chunk's column sums of phi(k)
          const float4 dz = reinterpret_cast<const float4 *>(smem + kOffZ + s * kZBytes)[lane];
          zl.x += dz.x;
          zl.y += dz.y;
          zl.z += dz.z;
          zl.w += dz.w;
          __syncwarp();  // every lane has read this chunk's z
          zw[lane] = zl;
          __syncwarp();
        }
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          uint4 uh, ul;
          split8(&qk[8 * c4], uh, ul);
          const int ch = 4 * (lane >> 4) + c4;
          sts128(phi + swz(row, ch), uh);
          sts128(plo + swz(row, ch), ul);
        }
      }
      {
        const uint32_t vt = smem_u32(smem + kOffStage + s * kStageBytes + kTileQ + kTileK);
        const uint32_t vhi = smem_u32(smem + kOffVt);
        const uint32_t vlo = vhi + kTileV;
        const int t = e >> 1, half = e & 1;
        const float r = gr.r[t];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t ch = 4 * half + k;
          float x[8];
          unpack8(lds128(vt + swz(t, ch)), x);
          if (!kNla) {  // r = 1 without gates
#pragma unroll
            for (int i = 0; i < 8; ++i) x[i] *= r;
          }
          uint4 uh, ul;
          split8(x, uh, ul);
          sts128(vhi + swz(t, ch), uh);
          sts128(vlo + swz(t, ch), ul);
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(&bars->p_ready[tb]);
    }
    if (kNla && q4 == 2 && vblk == 0 && p.nla_zT && !*abort)
      reinterpret_cast<float4 *>(p.nla_zT + ((size_t)b * p.H + h) * kDK)[lane] = zl;
  } else if (warp < 10) {
    // ============ warpgroup B: the state chain and the outputs ============
    const int q4 = warp & 3;
    const int srow = 32 * q4 + lane;      // d_k row of the state held by this thread
    const bool has_tok = lane < 16;
    const int tok = 16 * q4 + lane;
    const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
    // 2^g_C of the chunk and 2^g of this thread's token, read from the gate
    // ring before the slot can be refilled (the refill needs Q S of the chunk,
    // which waits for this warpgroup's o_free of the previous chunk)
    float egC = 1.f, eg_tok = 1.f;
    auto read_gates = [&](int c) -> bool {
      const int s = c % kStages;
      if (!wait_bar_warp<!kNla>(&bars->full[s], (uint32_t)(c / kStages) & 1u, abort)) return false;
      egC = ring[s].egC;
      eg_tok = ring[s].eg[tok & (kC - 1)];
      return true;
    };

    // the state slice S[srow, vblk*64 .. +64) in fp32 registers
    float S[kBV];
    {
      const float *src = p.S0 ? p.S0 + (((size_t)b * p.H + h) * kDK + srow) * p.DV + vblk * kBV : nullptr;
#pragma unroll
      for (int j = 0; j < kBV; j += 4) {
        const float4 v4 = src ? *reinterpret_cast<const float4 *>(src + j) : make_float4(0.f, 0.f, 0.f, 0.f);
        S[j] = v4.x; S[j + 1] = v4.y; S[j + 2] = v4.z; S[j + 3] = v4.w;
      }
    }
    auto write_state = [&](int sb) {
      const uint32_t hi = smem_u32(smem + kOffS + sb * 2 * kTileS);
      const uint32_t lo = hi + kTileS;
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) {
        uint4 uh, ul;
        split8(&S[8 * ch], uh, ul);
        sts128(hi + swz(srow, ch), uh);
        sts128(lo + swz(srow, ch), ul);
      }
      fence_proxy_async_smem();
      mbar_arrive(&bars->s_ready[sb]);
    };
    bool ok = read_gates(0);
    if (ok) write_state(0);
    for (int c = 0; c < nchunks && ok; ++c) {
      const int tb = c & 1;
      const uint32_t ph = (uint32_t)(c >> 1) & 1u;
      const int t0 = c * kC;

      // ---- S <- gamma_C S + K^T V~ (the hi and lo column halves summed) -------
      if (!wait_bar_warp<!kNla>(&bars->ds_ready, (uint32_t)c & 1u, abort)) { ok = false; break; }
      tc_fence_after();
      {
        const float gam = egC;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float dh[32], dl[32];
          tmem_ld32x2(tmem + kColDS + 32 * half + lane_base, tmem + kColDS + kBV + 32 * half + lane_base, dh, dl);
#pragma unroll
          for (int jj = 0; jj < 32; jj += 2) {
            if constexpr (kNla) {  // two-lane arithmetic: faster in this instance, slower in the gated ones
              const float2 r = __ffma2_rn(make_float2(gam, gam), make_float2(S[32 * half + jj], S[32 * half + jj + 1]),
                                          __fadd2_rn(make_float2(dh[jj], dh[jj + 1]), make_float2(dl[jj], dl[jj + 1])));
              S[32 * half + jj] = r.x;
              S[32 * half + jj + 1] = r.y;
            } else {
              S[32 * half + jj] = gam * S[32 * half + jj] + (dh[jj] + dl[jj]);
              S[32 * half + jj + 1] = gam * S[32 * half + jj + 1] + (dh[jj + 1] + dl[jj + 1]);
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&bars->ds_free);
      if (c + 1 < nchunks) write_state((c + 1) & 1);
      if (kEmit && ((c + 1) * kC) % p.state_every == 0 && (c + 1) * kC <= T) {
        // the state after this chunk closes a block: this thread's row slice goes out
        float *dst = p.S_blocks +
                     ((((size_t)b * p.nblocks + (c + 1) * kC / p.state_every - 1) * p.H + h) * kDK + srow) * p.DV +
                     vblk * kBV;
#pragma unroll
        for (int j = 0; j < kBV; j += 4)
          *reinterpret_cast<float4 *>(dst + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
      }

      // ---- o = gamma_i (Q S) + P V ----------------------------------------------
      if (!wait_bar_warp<!kNla>(&bars->o_ready[tb], ph, abort)) { ok = false; break; }
      float inv_den = 1.f;
      if (kNla) {
        const int ds = c & (kDenSlots - 1);
        if (!wait_bar_warp<!kNla>(&bars->den_ready[ds], (uint32_t)(c / kDenSlots) & 1u, abort)) { ok = false; break; }
        inv_den = reinterpret_cast<const float *>(smem + kOffDen)[ds * kC + (tok & (kC - 1))];
      }
      tc_fence_after();
      {
        const float gi = eg_tok;
        const int t = t0 + tok;
        const bool store = has_tok && t < T;
        const size_t obase = (((size_t)b * T + t) * p.H + h) * p.DV + vblk * kBV;
#pragma unroll
        for (int qt = 0; qt < 4; ++qt) {
          float o1[16], o1l[16], o2[16];
          tmem_ld16x3(tmem + kColO1 + 16 * qt + lane_base, tmem + kColO1 + kBV + 16 * qt + lane_base,
                      tmem + kColO2 + tb * 64 + 16 * qt + lane_base, o1, o1l, o2);
          float ov[16];
#pragma unroll
          for (int jj = 0; jj < 16; jj += 2) {
            if constexpr (kNla) {
              const float2 r = __ffma2_rn(make_float2(gi, gi),
                                          __fadd2_rn(make_float2(o1[jj], o1[jj + 1]), make_float2(o1l[jj], o1l[jj + 1])),
                                          make_float2(o2[jj], o2[jj + 1]));
              ov[jj] = r.x;
              ov[jj + 1] = r.y;
            } else {
              ov[jj] = gi * (o1[jj] + o1l[jj]) + o2[jj];
              ov[jj + 1] = gi * (o1[jj + 1] + o1l[jj + 1]) + o2[jj + 1];
            }
          }
          if (kNla) {
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) ov[jj] *= inv_den;
          }
          if (store) {
            if (kOutBf16) {
              uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(p.o) + obase + 16 * qt);
#pragma unroll
              for (int k = 0; k < 2; ++k) {
                uint32_t pk[4];
#pragma unroll
                for (int m = 0; m < 4; ++m)
                  pk[m] = bits(__floats2bfloat162_rn(ov[8 * k + 2 * m], ov[8 * k + 2 * m + 1]));
                dst[k] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
              }
            } else {
              float4 *dst = reinterpret_cast<float4 *>(reinterpret_cast<float *>(p.o) + obase + 16 * qt);
#pragma unroll
              for (int k = 0; k < 4; ++k)
                dst[k] = make_float4(ov[4 * k], ov[4 * k + 1], ov[4 * k + 2], ov[4 * k + 3]);
            }
          }
        }
      }
      if (c + 1 < nchunks && !read_gates(c + 1)) { ok = false; break; }
      tc_fence_before();
      mbar_arrive(&bars->o_free[tb]);
    }
    if (ok) {
      float *dst = p.S_T + (((size_t)b * p.H + h) * kDK + srow) * p.DV + vblk * kBV;
#pragma unroll
      for (int j = 0; j < kBV; j += 4)
        *reinterpret_cast<float4 *>(dst + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
    }
  } else {
    // ============ MMA issuer B: Q K^T (one chunk ahead) and P V ============
    if (lane == 0) {
      constexpr uint32_t id_qk = idesc_bf16(64, 64, false, false);  // Q K^T
      constexpr uint32_t id_pv = idesc_bf16(64, kBV, false, true);  // P V
      const uint32_t sbase = smem_u32(smem);
      const uint64_t dP = desc_sw128(sbase + kOffP, 16, 1024);
      // Q K^T of chunk c: M = 64 tokens, N = 64 tokens, K = d_k (2 swizzle blocks x 4 steps)
      auto issue_qk = [&](int c) -> bool {
        const int s = c % kStages, tb = c & 1;
        if (!wait_bar<!kNla>(&bars->full[s], (uint32_t)(c / kStages) & 1u, abort)) return false;
        if (!wait_bar<!kNla>(&bars->qk_free[tb], ((uint32_t)(c >> 1) & 1u) ^ 1u, abort)) return false;
        tc_fence_after();
        const uint32_t aQ = sbase + kOffStage + s * kStageBytes;
        const uint64_t dQ = desc_sw128(aQ, 16, 1024), dK = desc_sw128(aQ + kTileQ, 16, 1024);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t off = ((ks >> 2) * (kTileQ / 2) + (ks & 3) * 32) >> 4;
          umma_bf16(tmem + kColQK + tb * 64, dQ + off, dK + off, id_qk, ks > 0);
        }
        umma_commit(&bars->qk_ready[tb]);
        return true;
      };
      bool ok = issue_qk(0);
      for (int c = 0; c < nchunks && ok; ++c) {
        const int s = c % kStages;
        const int tb = c & 1;
        const uint32_t ph = (uint32_t)(c >> 1) & 1u;
        if (c + 1 < nchunks && !issue_qk(c + 1)) break;
        if (!wait_bar<!kNla>(&bars->p_ready[tb], ph, abort)) break;
        if (!wait_bar<!kNla>(&bars->o_free[tb], ph ^ 1u, abort)) break;   // P V buffer tb
        tc_fence_after();
        const uint64_t dV = desc_sw128(sbase + kOffStage + s * kStageBytes + kTileQ + kTileK, 16, 1024);
        // O2 = (Phi + Plo) V: M = 64, N = 64, K = 64 tokens
#pragma unroll
        for (int part = 0; part < 2; ++part)
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            umma_bf16(tmem + kColO2 + tb * 64, dP + ((part * kTileP + ks * 32) >> 4),
                      dV + ((ks * 2048) >> 4), id_pv, (part | ks) != 0);
        umma_commit(&bars->o_ready[tb]);
        umma_commit(&bars->p_free);   // P may be rewritten
        umma_commit(&bars->empty[s]);  // Q, K (Q K^T) and V of this stage are read
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (*abort && tid == 0 && p.dev_status) atomicOr(p.dev_status, GLINATTN_DEV_WAIT_TIMEOUT);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmCols);
  }
}

// ---- host side ----------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return (EncodeTiledFn) nullptr;
    return (EncodeTiledFn)f;
  }();
  return fn;
}

}  // namespace

// [B, T, H, d] bf16 activations as a 4-D map (d, H, T, B), box 64 x 1 x 64 x 1.
bool make_act_map(CUtensorMap *m, const void *base, int B, int T, int H, int d) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)B};
  const cuuint64_t strides[3] = {(cuuint64_t)d * 2, (cuuint64_t)H * d * 2, (cuuint64_t)T * H * d * 2};
  const cuuint32_t box[4] = {64, 1, (cuuint32_t)kC, 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_3d_map(CUtensorMap *m, const void *base, CUtensorMapDataType type, int elem_bytes,
                   const long long dims[3], const int box[3], bool swizzle) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t gd[3] = {(cuuint64_t)dims[0], (cuuint64_t)dims[1], (cuuint64_t)dims[2]};
  const cuuint64_t st[2] = {(cuuint64_t)dims[0] * elem_bytes, (cuuint64_t)dims[0] * dims[1] * elem_bytes};
  const cuuint32_t bx[3] = {(cuuint32_t)box[0], (cuuint32_t)box[1], (cuuint32_t)box[2]};
  const cuuint32_t es[3] = {1, 1, 1};
  return enc(m, type, 3, const_cast<void *>(base), gd, st, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_rows_map(CUtensorMap *m, const void *base, CUtensorMapDataType type, int elem_bytes,
                     int inner, int rows, int planes, int box_inner, bool swizzle) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)rows, (cuuint64_t)planes};
  const cuuint64_t strides[2] = {(cuuint64_t)inner * elem_bytes, (cuuint64_t)rows * inner * elem_bytes};
  const cuuint32_t box[3] = {(cuuint32_t)box_inner, (cuuint32_t)kC, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return enc(m, type, 3, const_cast<void *>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool prefill_tc_available() { return encode_fn() != nullptr; }

bool prefill_tc_supports(const glinattn_prefill_args &a) {
  return a.variant == GLINATTN_GLA && a.in_dtype == GLINATTN_BF16 && a.dk == kDK &&
         (a.dv == kDK || a.dv == kBV) && a.conv_w == nullptr && !a.qk_l2norm && a.seqlen > 0;
}

glinattn_status launch_prefill_tc(const glinattn_prefill_args &a, cudaStream_t stream) {
  return launch_prefill_tc_skip(a, stream, nullptr);
}

glinattn_status launch_prefill_tc_skip(const glinattn_prefill_args &a, cudaStream_t stream, const int *skip) {
  return launch_prefill_tc_nla(a, stream, skip, nullptr, nullptr, nullptr);
}

glinattn_status launch_prefill_tc_nla(const glinattn_prefill_args &a, cudaStream_t stream, const int *skip,
                                      const float *nla_dz, const float *nla_z0, float *nla_zT) {
  CUtensorMap tq, tk, tv;
  const int Hq = a.qk_heads > 0 ? a.qk_heads : a.heads;
  if (!make_act_map(&tq, a.q, a.batch, a.seqlen, Hq, kDK) ||
      !make_act_map(&tk, a.k, a.batch, a.seqlen, Hq, kDK) ||
      !make_act_map(&tv, a.v, a.batch, a.seqlen, a.heads, a.dv))
    return GLINATTN_ERR_CUDA;
  GlaParams p;
  p.rep = a.heads / Hq;
  p.DV = a.dv;
  p.skip = skip;
  p.B = a.batch;
  p.T = a.seqlen;
  p.H = a.heads;
  p.nchunks = (a.seqlen + kC - 1) / kC;
  p.out_bf16 = a.out_dtype == GLINATTN_BF16;
  p.alpha = a.alpha;
  p.S0 = a.S0;
  p.S_T = a.S_T;
  p.o = a.o;
  p.dev_status = a.dev_status;
  p.state_every = a.state_every > 0 && a.seqlen / a.state_every > 0 ? a.state_every : 0;
  p.nblocks = p.state_every ? a.seqlen / p.state_every : 0;
  p.S_blocks = a.S_blocks;
  p.nla_dz = nla_dz;
  p.nla_z0 = nla_z0;
  p.nla_zT = nla_zT;
  auto kernel = nla_dz ? (p.out_bf16 ? gla_prefill_kernel<true, false, true> : gla_prefill_kernel<false, false, true>)
                : p.out_bf16 ? (p.state_every ? gla_prefill_kernel<true, true, false> : gla_prefill_kernel<true, false, false>)
                             : (p.state_every ? gla_prefill_kernel<false, true, false> : gla_prefill_kernel<false, false, false>);
  const uint32_t smem_bytes = nla_dz ? kSmemBytesNla : kSmemBytes;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes) != cudaSuccess)
    return GLINATTN_ERR_CUDA;
  const unsigned grid = (unsigned)a.batch * (unsigned)a.heads * (unsigned)(a.dv / kBV);
  kernel<<<grid, kThreads, smem_bytes, stream>>>(tq, tk, tv, p);
  return cudaGetLastError() == cudaSuccess ? GLINATTN_OK : GLINATTN_ERR_CUDA;
}

}  // namespace glinattn
