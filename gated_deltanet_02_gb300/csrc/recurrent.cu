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
// The columns of S evolve independently (both updates left-multiply S by a
// matrix of k, alpha, beta only), so one CTA owns one column slice of one
// (request, head) state: the 128 x 64 half for d = 128, the whole state for
// smaller heads.  The slice is fetched into shared memory by one TMA tile
// load issued as soon as the slot id is known, while the threads run the
// front end (short convolution, L2 norm); each CTA needs 44 KB of shared
// memory at d = 128, so five slices per SM are in flight.  Thread (rg, cg)
// owns rows rg + ROWG*i of column group cg (4 consecutive columns, one
// 16-byte vector): every warp access to a state row is contiguous.  k S and
// q S are reduced in one pass, across row groups through shared memory in a
// fixed order (deterministic, no atomics).  Decode (1 step, in place) and
// speculative decode (D steps, a write after each) run this same code, so a
// draft state equals the state of repeated decode steps bit for bit.
#include <string.h>

#include "common.cuh"
#include "frontend.cuh"
#include "prefill_tc.cuh"
#include "sm100.cuh"

namespace glinattn {
namespace {

using namespace sm100;

template <int DK, int DV>
struct Shape {
  static constexpr int NSPLIT = DV == 128 ? 2 : 1;  // column slices per state
  static constexpr int DC = DV / NSPLIT;             // columns per CTA
  static constexpr int NT = DK == 128 ? 128 : ((DK * DV / 4 < 256) ? DK * DV / 4 : 256);
  static constexpr int COLG = DC / 4;               // 16-byte column groups
  static constexpr int ROWG = NT / COLG;            // row groups
  static constexpr int RPT = DK / ROWG;             // rows per thread
  static constexpr int NCH = 2 * DK + DC;           // front-end channels: q, k, own v slice
  static_assert(RPT >= 1 && ROWG * RPT == DK, "shape");
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

// phi(x) = elu(x) + 1, the positive feature map of normalised linear attention
__device__ __forceinline__ float feature_map(float x) { return x > 0.f ? x + 1.f : expf(x); }

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// kVar: the variant (GLINATTN_GLA or GLINATTN_GDN) as a template parameter, so
// each instance carries only its own update path; kAnyVariant reads it at run
// time (normalised linear attention, measured faster that way).
constexpr int kAnyVariant = -1;

template <int DK, int DV, int kVar>
__global__ void __launch_bounds__(Shape<DK, DV>::NT)
    recurrent_kernel(const __grid_constant__ CUtensorMap tstate, const RecurParams p) {
  using Sh = Shape<DK, DV>;
  constexpr int NW = (Sh::NT + 31) / 32;
  static_assert(Sh::NT >= DK && Sh::NT % 32 == 0 && (NW & (NW - 1)) == 0,
                "the L2 norm's pairwise sum wants one q and one k channel per thread and 2^m warps");
  constexpr int NCH = Sh::NCH;
  constexpr int MAXC = (NCH + Sh::NT - 1) / Sh::NT;  // front-end channels per thread
  constexpr uint32_t kSliceBytes = DK * Sh::DC * 4;
  const int half = blockIdx.x % Sh::NSPLIT;
  const int unit = blockIdx.x / Sh::NSPLIT;
  const int n = unit / p.H, h = unit - n * p.H;
  const int tid = threadIdx.x;
  const int cg = tid % Sh::COLG, rg = tid / Sh::COLG;
  const int col0 = half * Sh::DC;  // first state column of this CTA
  const size_t DD = (size_t)DK * DV;
  const int hq = h / (p.H / p.Hq);  // the q / k head (group) of head h
  const bool nla = kVar == kAnyVariant && p.variant == GLINATTN_NLA;  // no gates; phi(q), phi(k); z
  const bool gdn = kVar == kAnyVariant ? p.variant == GLINATTN_GDN : kVar == GLINATTN_GDN;

  extern __shared__ __align__(128) float4 s_state4[];  // DK rows x DC columns, row-major
  __shared__ float s_act[NCH];                          // q | k | own v slice after the front end
  __shared__ float s_red[Sh::ROWG][2][Sh::DC];
  __shared__ float s_wsum[2][NW];
  __shared__ float s_qk;
  __shared__ float s_z[DK];  // normalised linear attention: the normaliser z
  __shared__ float s_qz;     // and phi(q) . z before this step's update
  __shared__ int s_bad;
  __shared__ __align__(8) uint64_t s_bar;

  // global channel of local front-end channel c: q (0..DK-1), k (DK..2DK-1), own v slice
  auto chan = [&](int c) {
    if (c < 2 * DK) return (c / DK) * p.H * DK + h * DK + (c % DK);
    return 2 * p.H * DK + h * DV + col0 + (c - 2 * DK);
  };
  // input element of local channel c for token row `row` (index of (n, t, h));
  // q and k rows are indexed by (n, t, hq)
  auto act_at = [&](int c, size_t row) {
    if (c >= 2 * DK) return load_act(p.v, row * DV + col0 + (c - 2 * DK), p.in_bf16);
    const size_t rq = (row / p.H) * p.Hq + hq;
    return load_act(c < DK ? p.q : p.k, rq * DK + (c % DK), p.in_bf16);
  };
  // conv-cache channels written by this CTA: q and k by slice 0, each v slice by its owner
  auto writes_chan = [&](int c) { return c >= 2 * DK || half == 0; };

  // steps applied by this request: all, or its accepted length (replay)
  int steps_n = p.steps;
  if (p.step_count) {
    steps_n = p.step_count[n];
    if (steps_n < 0 || steps_n > p.steps) {
      if (tid == 0 && half == 0 && p.dev_status) atomicOr(p.dev_status, GLINATTN_DEV_BAD_COUNT);
      return;
    }
    if (steps_n == 0) return;  // nothing accepted: the slot stays as it is
  }
  // ---- every independent load is issued first ----------------------------------
  int slot = n;
  bool slot_ok = true;
  if (p.src_slot) {
    slot = p.src_slot[n];
    slot_ok = !(p.pool_slots > 0 && (slot < 0 || slot >= p.pool_slots));
  }
  const bool has_src = p.S_src != nullptr && slot_ok;
  if (tid == 0) {
    mbar_init(&s_bar, 1);
    fence_mbar_init();
    if (has_src) {
      mbar_arrive_expect_tx(&s_bar, kSliceBytes);
      tma_load_3d(s_state4, &tstate, &s_bar, col0, 0, slot * p.H + h);
    }
    s_bad = 0;
  }
  const bool conv = p.conv_w != nullptr;
  // gates and destination slot of step 0 (prefetched one step ahead afterwards)
  float a_next = 1.f, b_next = 0.f;
  int dslot_next = n;
  if (p.steps > 0) {
    const size_t row0 = ((size_t)n * p.steps) * p.H + h;
    a_next = nla ? 1.f : p.alpha[row0];
    if (gdn) b_next = p.beta[row0];
    if (p.dst_slot) dslot_next = p.dst_slot[(size_t)n * (p.dst_per_step ? p.steps : 1)];
  }
  float xr[MAXC], wr[MAXC][4], hr[MAXC][3];
  {
    const size_t row0 = ((size_t)n * p.steps) * p.H + h;
#pragma unroll
    for (int i = 0; i < MAXC; ++i) {
      const int c = tid + i * Sh::NT;
      xr[i] = 0.f;
      wr[i][0] = wr[i][1] = wr[i][2] = 0.f;
      wr[i][3] = 1.f;
      hr[i][0] = hr[i][1] = hr[i][2] = 0.f;
      if (c < NCH) {
        if (p.steps > 0) xr[i] = act_at(c, row0);
        if (conv) {
          const float4 w = *reinterpret_cast<const float4 *>(p.conv_w + (size_t)chan(c) * 4);
          wr[i][0] = w.x; wr[i][1] = w.y; wr[i][2] = w.z; wr[i][3] = w.w;
          if (p.conv_src && slot_ok)
#pragma unroll
            for (int j = 0; j < 3; ++j)
              hr[i][j] = load_act(p.conv_src, ((size_t)slot * 3 + j) * p.Cch + chan(c), p.in_bf16);
        }
      }
    }
  }
  // ---- unit validation: slots in range, gates in (0, 1] --------------------------
  int bad = slot_ok ? 0 : GLINATTN_DEV_BAD_SLOT;
  if (p.pool_slots > 0 && p.dst_slot) {
    const int nd = p.dst_per_step ? p.steps : 1;
    for (int t = tid; t < nd; t += Sh::NT) {
      const int s = p.dst_slot[(size_t)n * nd + t];
      if (s < 0 || s >= p.pool_slots) bad |= GLINATTN_DEV_BAD_SLOT;
    }
  }
  for (int t = tid; t < steps_n && !nla; t += Sh::NT) {
    const float a = p.alpha[((size_t)n * p.steps + t) * p.H + h];
    if (!(a > 0.f && a <= 1.f)) bad |= GLINATTN_DEV_BAD_GATE;
  }
  __syncthreads();  // s_bad initialised, barrier initialised
  if (bad) atomicOr(&s_bad, bad);
  __syncthreads();
  if (s_bad) {
    if (has_src) mbar_wait(&s_bar, 0);  // let the copy land before the CTA exits
    if (tid == 0 && half == 0 && p.dev_status) atomicOr(p.dev_status, (uint32_t)s_bad);
    return;
  }
  if (!has_src) {
#pragma unroll
    for (int i = 0; i < Sh::RPT; ++i)
      s_state4[(rg + Sh::ROWG * i) * Sh::COLG + cg] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  if (nla)  // read by warp 0 after the first step's barrier
    for (int i = tid; i < DK; i += Sh::NT)
      s_z[i] = p.z_src && slot_ok ? p.z_src[((size_t)slot * p.H + h) * DK + i] : 0.f;
  // The slices of one state share the q / k conv history, and slice 0 writes it
  // back (in place for decode): every slice has read it before any writes it.
  bool history_released = Sh::NSPLIT == 1;
  auto release_history = [&]() {
    if (!history_released) {
      cluster_wait();
      history_released = true;
    }
  };
  if (Sh::NSPLIT > 1) cluster_arrive();

  for (int t = 0; t < steps_n; ++t) {
    const size_t row = ((size_t)n * p.steps + t) * p.H + h;  // (n, t, h)
    const float a = a_next, bgate = b_next;
    const int dslot_t = dslot_next;
    if (t + 1 < steps_n) {
      a_next = nla ? 1.f : p.alpha[row + p.H];
      if (gdn) b_next = p.beta[row + p.H];
      if (p.dst_slot && p.dst_per_step) dslot_next = p.dst_slot[(size_t)n * p.steps + t + 1];
    }
    // ---- front end in registers: conv, history shift, next token prefetch -------
    float yv[MAXC];
    float sq = 0.f, sk = 0.f;
#pragma unroll
    for (int i = 0; i < MAXC; ++i) {
      const int c = tid + i * Sh::NT;
      const float x = xr[i];
      float y = conv ? fe::conv4(wr[i][0], wr[i][1], wr[i][2], wr[i][3], hr[i][0], hr[i][1], hr[i][2], x) : x;
      if (nla && c < 2 * DK) y = feature_map(y);
      yv[i] = y;
      // at most one q and one k channel per thread (NT >= DK)
      if (c < DK) sq = __fmul_rn(y, y);
      else if (c < 2 * DK) sk = __fmul_rn(y, y);
      hr[i][0] = hr[i][1];
      hr[i][1] = hr[i][2];
      hr[i][2] = x;
      if (c < NCH && t + 1 < steps_n) xr[i] = act_at(c, row + p.H);
    }
    float iq = 1.f, ik = 1.f;
    if (p.qk_l2norm) {  // pairwise sums of squares: lanes, then warps
      sq = fe::warp_pairwise_sum(sq);
      sk = fe::warp_pairwise_sum(sk);
      if ((tid & 31) == 0) {
        s_wsum[0][tid >> 5] = sq;
        s_wsum[1][tid >> 5] = sk;
      }
      __syncthreads();
      iq = fe::inv_norm(fe::pairwise_sum<NW>(s_wsum[0]));
      ik = fe::inv_norm(fe::pairwise_sum<NW>(s_wsum[1]));
    }
    const bool round_act = p.in_bf16 && (conv || p.qk_l2norm || nla);
#pragma unroll
    for (int i = 0; i < MAXC; ++i) {
      const int c = tid + i * Sh::NT;
      if (c < NCH) {
        float y = yv[i];
        if (c < DK) y = __fmul_rn(y, iq);
        else if (c < 2 * DK) y = __fmul_rn(y, ik);
        s_act[c] = round_act ? round_bf16(y) : y;
      }
    }
    if (t == 0 && has_src) {  // the state copy must have landed
      const bool ok = mbar_wait(&s_bar, 0);
      if (!__syncthreads_and(ok)) {
        if (tid == 0 && p.dev_status) atomicOr(p.dev_status, GLINATTN_DEV_WAIT_TIMEOUT);
        release_history();
        return;
      }
    } else {
      __syncthreads();
    }

    // ---- q.k (one warp, fixed order) and the partial k S, q S ------------------
    if (tid < 32) {
      float acc = 0.f, accz = 0.f;
      for (int i = tid; i < DK; i += 32) {
        acc += s_act[i] * s_act[DK + i];
        if (nla) accz += s_act[i] * s_z[i];
      }
      acc = warp_sum(acc);
      if (nla) accz = warp_sum(accz);
      if (tid == 0) {
        s_qk = acc;
        s_qz = accz;
      }
    }
    const float *sqa = s_act, *ska = s_act + DK, *sva = s_act + 2 * DK;
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f), y = x;
#pragma unroll
    for (int i = 0; i < Sh::RPT; ++i) {
      const int r = rg + Sh::ROWG * i;
      const float4 S = s_state4[r * Sh::COLG + cg];
      const float kr = ska[r], qr = sqa[r];
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
    const float4 vv = *reinterpret_cast<const float4 *>(sva + 4 * cg);
    float4 u = vv;
    if (gdn) {
      const float b = bgate;
      u.x = b * (vv.x - a * x.x);
      u.y = b * (vv.y - a * x.y);
      u.z = b * (vv.z - a * x.z);
      u.w = b * (vv.w - a * x.w);
    }
    const bool last = (t == steps_n - 1);
    const bool emit = p.S_dst && (p.dst_per_step || last);
    float *dst = nullptr;
    const size_t dslot = (size_t)dslot_t;
    if (emit) dst = p.S_dst + (dslot * p.H + h) * DD + col0;
    float *bdst = nullptr;  // prefill state emitted at a block boundary
    if (p.state_every && (t + 1) % p.state_every == 0)
      bdst = p.S_blocks + (((size_t)n * p.nblocks + (t + 1) / p.state_every - 1) * p.H + h) * DD + col0;
#pragma unroll
    for (int i = 0; i < Sh::RPT; ++i) {
      const int r = rg + Sh::ROWG * i;
      const float kr = ska[r];
      float4 S = s_state4[r * Sh::COLG + cg];
      S.x = a * S.x + kr * u.x;
      S.y = a * S.y + kr * u.y;
      S.z = a * S.z + kr * u.z;
      S.w = a * S.w + kr * u.w;
      if (!last) s_state4[r * Sh::COLG + cg] = S;
      if (emit) *reinterpret_cast<float4 *>(dst + (size_t)r * DV + 4 * cg) = S;
      if (bdst) *reinterpret_cast<float4 *>(bdst + (size_t)r * DV + 4 * cg) = S;
    }
    if (nla && tid < DK) {  // z <- z + phi(k); every reader of the old z is past the barrier
      s_z[tid] += ska[tid];
      if (emit && half == 0 && p.z_dst) {
        release_history();  // the other slice has read the source normaliser (it may be this slot)
        p.z_dst[(dslot * p.H + h) * DK + tid] = s_z[tid];
      }
    }
    if (rg == 0 && p.o) {
      const float qk = s_qk;
      // normalised linear attention divides by phi(q) . z_t = phi(q) . z_{t-1} + phi(q) . phi(k)
      const float inv = nla ? 1.f / (s_qz + qk + 1e-6f) : 1.f;
      const size_t ob = row * DV + col0 + 4 * cg;
      store_act(p.o, ob + 0, (a * y.x + qk * u.x) * inv, p.out_bf16);
      store_act(p.o, ob + 1, (a * y.y + qk * u.y) * inv, p.out_bf16);
      store_act(p.o, ob + 2, (a * y.z + qk * u.z) * inv, p.out_bf16);
      store_act(p.o, ob + 3, (a * y.w + qk * u.w) * inv, p.out_bf16);
    }
    if (emit && conv && p.conv_dst) {
      release_history();
#pragma unroll
      for (int i = 0; i < MAXC; ++i) {
        const int c = tid + i * Sh::NT;
        if (c < NCH && writes_chan(c))
#pragma unroll
          for (int j = 0; j < 3; ++j)
            store_act(p.conv_dst, (dslot * 3 + j) * p.Cch + chan(c), hr[i][j], p.in_bf16);
      }
    }
  }

  if (p.steps == 0) {  // a zero-length segment hands its inputs straight on
    if (has_src && !__syncthreads_and(mbar_wait(&s_bar, 0))) {
      if (tid == 0 && p.dev_status) atomicOr(p.dev_status, GLINATTN_DEV_WAIT_TIMEOUT);
      release_history();
      return;
    }
    __syncthreads();
    release_history();
    float *dst = p.S_dst + ((size_t)n * p.H + h) * DD + col0;
#pragma unroll
    for (int i = 0; i < Sh::RPT; ++i) {
      const int r = rg + Sh::ROWG * i;
      *reinterpret_cast<float4 *>(dst + (size_t)r * DV + 4 * cg) = s_state4[r * Sh::COLG + cg];
    }
    if (conv && p.conv_dst) {
#pragma unroll
      for (int i = 0; i < MAXC; ++i) {
        const int c = tid + i * Sh::NT;
        if (c < NCH && writes_chan(c))
#pragma unroll
          for (int j = 0; j < 3; ++j)
            store_act(p.conv_dst, ((size_t)n * 3 + j) * p.Cch + chan(c), hr[i][j], p.in_bf16);
      }
    }
    if (nla && half == 0 && p.z_dst)
      for (int i = tid; i < DK; i += Sh::NT) p.z_dst[((size_t)n * p.H + h) * DK + i] = s_z[i];
  }
  release_history();
}

template <int DK, int DV, int kVar>
cudaError_t launch_variant(const RecurParams &p, cudaStream_t stream) {
  using Sh = Shape<DK, DV>;
  const unsigned grid = (unsigned)p.N * (unsigned)p.H * Sh::NSPLIT;
  constexpr int smem = DK * Sh::DC * 4;
  CUtensorMap tmap;
  memset(&tmap, 0, sizeof(tmap));
  if (p.S_src) {
    // the state source as (columns, rows, slot * H + head) planes; box = one column slice
    const long long planes = (long long)(p.src_slot ? p.pool_slots : p.N) * p.H;
    const long long dims[3] = {DV, DK, planes};
    const int box[3] = {Sh::DC, DK, 1};
    if (!encode_3d_map(&tmap, p.S_src, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, dims, box, false))
      return cudaErrorInvalidValue;
  }
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(recurrent_kernel<DK, DV, kVar>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(Sh::NT);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = Sh::NSPLIT;  // the slices of one state run as one cluster
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, recurrent_kernel<DK, DV, kVar>, tmap, p);
}

template <int DK, int DV>
cudaError_t launch(const RecurParams &p, cudaStream_t stream) {
  if (p.variant == GLINATTN_GDN) return launch_variant<DK, DV, GLINATTN_GDN>(p, stream);
  if (p.variant == GLINATTN_GLA) return launch_variant<DK, DV, GLINATTN_GLA>(p, stream);
  return launch_variant<DK, DV, kAnyVariant>(p, stream);
}

}  // namespace

glinattn_status launch_recurrent(const RecurParams &p, int dk, int dv, cudaStream_t stream) {
  if ((long long)p.N * p.H == 0) return GLINATTN_OK;
  if (dk == dv && verify128_supports(p, dk))
    return launch_verify128(p, stream) == cudaSuccess ? GLINATTN_OK : GLINATTN_ERR_CUDA;
  if (dk == dv && decode128_supports(p, dk))
    return launch_decode128(p, stream) == cudaSuccess ? GLINATTN_OK : GLINATTN_ERR_CUDA;
  cudaError_t e;
  if (dk == 128 && dv == 64) {
    e = launch<128, 64>(p, stream);
  } else if (dk != dv) {
    return GLINATTN_ERR_UNSUPPORTED;
  } else {
    switch (dk) {
      case 16: e = launch<16, 16>(p, stream); break;
      case 32: e = launch<32, 32>(p, stream); break;
      case 64: e = launch<64, 64>(p, stream); break;
      case 128: e = launch<128, 128>(p, stream); break;
      default: return GLINATTN_ERR_UNSUPPORTED;
    }
  }
  return e == cudaSuccess ? GLINATTN_OK : GLINATTN_ERR_CUDA;
}

}  // namespace glinattn
