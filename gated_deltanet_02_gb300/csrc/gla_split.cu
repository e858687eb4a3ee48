// gla_split.cu -- gated linear attention prefill split along the sequence, for
// calls with too few (batch, head, d_v slice) units to fill the GPU.
//
// "Inference for linear attention and hybrid architectures", section "Two
// ways to write the same computation": only the state passes from one chunk to
// the next, and with a scalar gate the state after a stretch of tokens is
//   S_end = Gamma S_start + S_local,
// where Gamma is the product of the stretch's gates and S_local the state the
// stretch reaches from a zero start.  So the sequence can be cut into P pieces
// of whole chunks that run side by side:
//
//   1. gla_state_kernel, one CTA per (piece, head, d_v slice): S_local and
//      Gamma of its piece, S_local as one accumulation of K^T diag(w) V over
//      the piece's chunks (w_t the decay from token t to the piece end; no
//      scores, no outputs, no chain through the state), and whether any gate
//      of the whole sequence is invalid;
//   2. gla_combine_kernel: S_start of every piece, serially over the P
//      pieces (one multiply-add per state element and piece), and S_T;
//   3. gla_prefill_kernel on the pieces as separate sequences, each from its
//      S_start: the outputs.
//
// Used when B * H * (d_v / 64) leaves more than half of the SMs idle and T
// splits into equal pieces of at least four chunks; otherwise the prefill
// runs unsplit.
#include <atomic>

#include <cuda.h>
#include <cuda_bf16.h>
#include <string.h>

#include "common.cuh"
#include "prefill_tc.cuh"
#include "sm100.cuh"
#include "tc_common.cuh"

namespace glinattn {
namespace {

using namespace sm100;
using namespace tc;

constexpr int kC = 64;     // chunk length
constexpr int kDK = 128;   // key head size
constexpr int kBV = 64;    // d_v columns per CTA
constexpr int kStages = 4;
constexpr int kPrefetch = 4;  // chunks prefetched into L2 beyond the shared-memory ring
constexpr int kThreads = 192;  // warp 0 TMA + weights, warp 1 MMA issuer, warps 2-5 V~ and the end state
constexpr uint32_t kTileK = kC * kDK * 2;   // 16 KiB: two 64-column swizzled blocks
constexpr uint32_t kTileV = kC * kBV * 2;   // 8 KiB
constexpr uint32_t kStageBytes = kTileK + kTileV;
constexpr uint32_t kOffStage = 0;
constexpr int kVtBufs = 2;                             // V~ [hi | lo] buffers
constexpr uint32_t kOffVt = kStages * kStageBytes;
constexpr uint32_t kOffG = kOffVt + kVtBufs * 2 * kTileV;  // weights [stage]: w[64]
constexpr uint32_t kGateFloats = kC + 4;
constexpr uint32_t kOffBar = kOffG + kStages * kGateFloats * 4;
constexpr uint32_t kSmemBytes = kOffBar + 256 + 1024;
constexpr uint32_t kTmCols = 128;  // S_local as K^T [V~hi | V~lo], one accumulator

struct StateParams {
  int BP, P, L, T, H, rep, DV, nchunks;  // BP = B * P sequences of L tokens
  const float *alpha;                      // [B, T, H] (the whole sequence)
  float *S_local;                          // [BP, H, dk, dv]
  float *gamma;                            // [BP, H]
  int *skip;                               // [BP, H]: 1 when a gate of the unit is invalid
  uint32_t *dev_status;
};

struct StateBars {
  uint64_t full[kStages], empty[kStages];
  uint64_t vt_ready[kVtBufs], vt_free[kVtBufs], ds_ready;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(StateBars) <= 256, "barrier block");

__global__ void __launch_bounds__(kThreads, 1)
    gla_state_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                     const StateParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  StateBars *bars = reinterpret_cast<StateBars *>(smem + kOffBar);
  float *gates = reinterpret_cast<float *>(smem + kOffG);
  volatile int *abort = &bars->abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nvb = p.DV / kBV;
  const int vblk = blockIdx.x % nvb;
  const int bph = blockIdx.x / nvb;                  // (piece sequence, head)
  const int bp = bph / p.H, h = bph - bp * p.H;
  const int b = bp / p.P;
  const int hq = h / p.rep;
  const int L = p.L, nchunks = p.nchunks;

  // ---- every gate of the whole sequence in (0, 1]: else the unit is skipped ------
  {
    int bad = 0;
    for (int t = tid; t < p.T; t += kThreads) {
      const float a = p.alpha[((size_t)b * p.T + t) * p.H + h];
      bad |= !(a > 0.f && a <= 1.f);
    }
    bad = __syncthreads_or(bad);
    if (tid == 0 && vblk == 0) p.skip[bph] = bad;
    if (bad) {
      if (tid == 0 && vblk == 0 && bp % p.P == 0 && p.dev_status) atomicOr(p.dev_status, GLINATTN_DEV_BAD_GATE);
      return;
    }
  }

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->full[s], 1 + 32);  // the TMA transaction and the 32 gate lanes
      mbar_init(&bars->empty[s], 1);
    }
    for (int i = 0; i < kVtBufs; ++i) {
      mbar_init(&bars->vt_ready[i], 128);
      mbar_init(&bars->vt_free[i], 1);
    }
    mbar_init(&bars->ds_ready, 1);
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
  const int tb0 = (bp % p.P) * L;  // first token of the piece in the whole sequence (for alpha)
  const size_t arow = (size_t)b * p.T;

  // The piece's end state from a zero start is a plain sum,
  //   S_local = sum_t w_t k_t^T v_t,  w_t = prod_{s > t in the piece} alpha_s,
  // so it is one accumulation of K^T [V~hi | V~lo] over all chunks (V~ = diag(w) V)
  // with no chain through the state.  The chunks are taken from the last to
  // the first, so w comes from a running suffix sum of log2 alpha.
  if (warp == 0) {
    // ============ TMA producer (lane 0) and the weights w of each chunk (all lanes) ============
    // chunk k of the loop (counted from the last) into L2, ahead of the ring
    auto prefetch = [&](int k) {
      if (k >= nchunks) return;
      const int t0 = (nchunks - 1 - k) * kC;
      tma_prefetch_l2_4d(&tk, 0, hq, t0, bp);
      tma_prefetch_l2_4d(&tk, 64, hq, t0, bp);
      tma_prefetch_l2_4d(&tv, vblk * kBV, h, t0, bp);
    };
    if (lane == 0) {
      prefetch_tensormap(&tk);
      prefetch_tensormap(&tv);
      for (int k = 0; k < kPrefetch; ++k) prefetch(kStages + k);
    }
    float gsuf = 0.f;  // sum of log2 alpha over the chunks after this one
    bool ok = true;
    // lane l: tokens 2l, 2l + 1 of a chunk; their gates are loaded one chunk
    // ahead, so the loads' latency does not sit in the chunk loop
    auto load_gates = [&](int c, float &x0, float &x1) {
      const int ta = c * kC + 2 * lane, tb = ta + 1;
      x0 = ta < L ? p.alpha[(arow + tb0 + ta) * p.H + h] : 1.f;
      x1 = tb < L ? p.alpha[(arow + tb0 + tb) * p.H + h] : 1.f;
    };
    float na0 = 1.f, na1 = 1.f;
    if (nchunks > 0) load_gates(nchunks - 1, na0, na1);
    for (int k = 0; k < nchunks; ++k) {
      const int c = nchunks - 1 - k, s = k % kStages;
      const float a0 = na0, a1 = na1;
      if (c > 0) load_gates(c - 1, na0, na1);
      if (lane == 0) prefetch(k + kStages + kPrefetch);
      const uint32_t use = (uint32_t)(k / kStages);
      if (!wait_bar_warp(&bars->empty[s], (use & 1u) ^ 1u, abort)) { ok = false; break; }
      if (lane == 0) {
        uint8_t *st = smem + kOffStage + s * kStageBytes;
        mbar_arrive_expect_tx(&bars->full[s], kStageBytes);
        const int t0 = c * kC;
        tma_load_4d(st, &tk, &bars->full[s], 0, hq, t0, bp);
        tma_load_4d(st + kTileK / 2, &tk, &bars->full[s], 64, hq, t0, bp);
        tma_load_4d(st + kTileK, &tv, &bars->full[s], vblk * kBV, h, t0, bp);
      }
      // g = cumsum(log2 alpha) inside the chunk, w = 2^(gsuf + g_C - g)
      const float l0 = log2f(a0), l1 = log2f(a1);
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
      float *gr = gates + s * kGateFloats;
      gr[2 * lane] = exp2f(gsuf + (gC - ga));
      gr[2 * lane + 1] = exp2f(gsuf + (gC - gb));
      mbar_arrive(&bars->full[s]);  // releases this lane's weight writes
      gsuf += gC;
    }
    if (ok && lane == 0 && vblk == 0) p.gamma[bph] = exp2f(gsuf);  // the piece's total decay
  } else if (warp == 1) {
    // ============ MMA issuer: S_local += K^T [V~hi | V~lo], one accumulator ============
    if (lane == 0) {
      constexpr uint32_t id_ds = idesc_bf16(128, 2 * kBV, true, true);
      const uint32_t sbase = smem_u32(smem);
      bool ok = true;
      for (int k = 0; k < nchunks; ++k) {
        const int s = k % kStages, vb = k % kVtBufs;
        const uint32_t ph = (uint32_t)(k / kVtBufs) & 1u;
        if (!wait_bar(&bars->full[s], (uint32_t)(k / kStages) & 1u, abort) ||
            !wait_bar(&bars->vt_ready[vb], ph, abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t dKm = desc_sw128(sbase + kOffStage + s * kStageBytes, kTileK / 2, 1024);
        const uint64_t dVt = desc_sw128(sbase + kOffVt + vb * 2 * kTileV, kTileV, 1024);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          umma_bf16(tmem, dKm + ((ks * 2048) >> 4), dVt + ((ks * 2048) >> 4), id_ds, (k | ks) != 0);
        umma_commit(&bars->vt_free[vb]);
        umma_commit(&bars->empty[s]);
      }
      if (ok) umma_commit(&bars->ds_ready);
    }
  } else {
    // ============ warps 2-5: V~ = diag(w) V per chunk, then S_local from TMEM ============
    const int e = tid - 64;  // 0..127
    const int q4 = warp & 3;
    const int srow = 32 * q4 + lane;  // d_k row of the state held by this thread
    const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
    bool ok = true;
    for (int k = 0; k < nchunks && ok; ++k) {
      const int s = k % kStages, vb = k % kVtBufs;
      const uint32_t ph = (uint32_t)(k / kVtBufs) & 1u;
      if (!wait_bar_warp(&bars->full[s], (uint32_t)(k / kStages) & 1u, abort)) { ok = false; break; }
      if (!wait_bar_warp(&bars->vt_free[vb], ph ^ 1u, abort)) { ok = false; break; }
      const float *gr = gates + s * kGateFloats;
      const uint32_t vt = smem_u32(smem + kOffStage + s * kStageBytes + kTileK);
      const uint32_t vhi = smem_u32(smem + kOffVt + vb * 2 * kTileV), vlo = vhi + kTileV;
      const int t = e >> 1, half = e & 1;
      const float w = gr[t];
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint32_t ch = 4 * half + kk;
        float x[8];
        unpack8(lds128(vt + swz(t, ch)), x);
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] *= w;
        uint4 uh, ul;
        split8(x, uh, ul);
        sts128(vhi + swz(t, ch), uh);
        sts128(vlo + swz(t, ch), ul);
      }
      fence_proxy_async_smem();
      mbar_arrive(&bars->vt_ready[vb]);
    }
    if (ok && wait_bar_warp(&bars->ds_ready, 0u, abort)) {
      tc_fence_after();
      float *dst = p.S_local + (((size_t)bph * kDK) + srow) * p.DV + vblk * kBV;
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        float dh[32], dl[32];
        tmem_ld32x2(tmem + 32 * hf + lane_base, tmem + kBV + 32 * hf + lane_base, dh, dl);
#pragma unroll
        for (int j = 0; j < 32; j += 4)
          *reinterpret_cast<float4 *>(dst + 32 * hf + j) =
              make_float4(dh[j] + dl[j], dh[j + 1] + dl[j + 1], dh[j + 2] + dl[j + 2], dh[j + 3] + dl[j + 3]);
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

// S_start of every piece and the final state: per element of a (sequence,
// head) state, serially over the pieces.
// A unit with an invalid gate (skip set by the state pass) writes nothing.
__global__ void __launch_bounds__(256) gla_combine_kernel(int B, int P, int H, int DD, const float *S0,
                                                         const float *S_local, const float *gamma,
                                                         const int *skip, float *S_start, float *S_T) {
  const size_t e = (size_t)blockIdx.x * 256 + threadIdx.x;  // (b, h, element)
  const size_t per = (size_t)H * DD;
  if (e >= (size_t)B * per) return;
  const int b = (int)(e / per);
  const size_t he = e - (size_t)b * per;
  const int h = (int)(he / DD);
  if (skip[(size_t)b * P * H + h]) return;
  float s = S0 ? S0[e] : 0.f;
  for (int q = 0; q < P; ++q) {
    const size_t bp = (size_t)b * P + q;
    S_start[bp * per + he] = s;
    s = gamma[bp * H + h] * s + S_local[bp * per + he];
  }
  S_T[e] = s;
}

struct SplitPlan {
  int P, L;
};

// SMs of the current device, looked up once per device (the split decision,
// and so the queried scratch size, follows the device the call runs on).
int sm_count() {
  constexpr int kMaxDevices = 64;
  static std::atomic<int> cache[kMaxDevices];
  int dev = 0, v = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < kMaxDevices && (v = cache[dev].load(std::memory_order_relaxed)) > 0) return v;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < kMaxDevices) cache[dev].store(v, std::memory_order_relaxed);
  return v;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

struct SplitCarve {
  float *S_local, *S_start, *S_scratch, *gamma;
  int *skip;
  size_t bytes;
};

SplitCarve carve(void *base, const glinattn_prefill_args &a, int P) {
  const size_t st = align256((size_t)a.batch * P * a.heads * a.dk * a.dv * 4);
  const size_t g = align256((size_t)a.batch * P * a.heads * 4);
  uint8_t *p = static_cast<uint8_t *>(base);
  SplitCarve c;
  c.S_local = reinterpret_cast<float *>(p);
  c.S_start = reinterpret_cast<float *>(p + st);
  c.S_scratch = reinterpret_cast<float *>(p + 2 * st);
  c.gamma = reinterpret_cast<float *>(p + 3 * st);
  c.skip = reinterpret_cast<int *>(p + 3 * st + g);
  c.bytes = 3 * st + 2 * g;
  return c;
}

}  // namespace

// P pieces when the unsplit launch would leave more than half of the SMs idle,
// every piece a whole number of chunks and at least four of them; 1 otherwise.
int gla_split_pieces(const glinattn_prefill_args &a) {
  if (!prefill_tc_supports(a) || a.state_every != 0 || a.variant != GLINATTN_GLA) return 1;
  const int sms = sm_count();
  const long long units = (long long)a.batch * a.heads * (a.dv / kBV);
  if (sms <= 0 || units <= 0 || 2 * units > sms) return 1;
  int P = (int)(sms / units);
  if (P > 4) P = 4;
  for (; P >= 2; --P)
    if (a.seqlen % (P * kC) == 0 && a.seqlen / P >= 4 * kC && (long long)a.batch * P <= 65535) break;
  return P >= 2 ? P : 1;
}

size_t gla_split_workspace_bytes(const glinattn_prefill_args &a) {
  const int P = gla_split_pieces(a);
  return P > 1 ? carve(nullptr, a, P).bytes : 0;
}

glinattn_status launch_gla_split(const glinattn_prefill_args &a, cudaStream_t stream) {
  const int P = gla_split_pieces(a);
  const int B = a.batch, T = a.seqlen, H = a.heads, L = T / P;
  const int Hq = a.qk_heads > 0 ? a.qk_heads : H;
  const SplitCarve w = carve(a.workspace, a, P);
  // the pieces as B * P sequences of L tokens: the activations are contiguous in (b, t)
  CUtensorMap tk, tv;
  if (!make_act_map(&tk, a.k, B * P, L, Hq, kDK) || !make_act_map(&tv, a.v, B * P, L, H, a.dv))
    return GLINATTN_ERR_CUDA;
  StateParams sp;
  sp.BP = B * P;
  sp.P = P;
  sp.L = L;
  sp.T = T;
  sp.H = H;
  sp.rep = H / Hq;
  sp.DV = a.dv;
  sp.nchunks = L / kC;
  sp.alpha = a.alpha;
  sp.S_local = w.S_local;
  sp.gamma = w.gamma;
  sp.skip = w.skip;
  sp.dev_status = a.dev_status;
  if (cudaFuncSetAttribute(gla_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) !=
      cudaSuccess)
    return GLINATTN_ERR_CUDA;
  const unsigned grid = (unsigned)(B * P) * (unsigned)H * (unsigned)(a.dv / kBV);
  gla_state_kernel<<<grid, kThreads, kSmemBytes, stream>>>(tk, tv, sp);
  if (cudaGetLastError() != cudaSuccess) return GLINATTN_ERR_CUDA;
  const int DD = a.dk * a.dv;
  const size_t total = (size_t)B * H * DD;
  gla_combine_kernel<<<(unsigned)((total + 255) / 256), 256, 0, stream>>>(B, P, H, DD, a.S0, w.S_local, w.gamma,
                                                                         w.skip, w.S_start, a.S_T);
  if (cudaGetLastError() != cudaSuccess) return GLINATTN_ERR_CUDA;
  // the outputs: every piece from its start state; the pieces' end states are not needed
  glinattn_prefill_args g = a;
  g.batch = B * P;
  g.seqlen = L;
  g.S0 = w.S_start;
  g.S_T = w.S_scratch;
  return launch_prefill_tc_skip(g, stream, w.skip);
}

}  // namespace glinattn
