// decode128.cu -- persistent, pipelined decode and speculative decode for
// 128 x 128 fp32 head states held in a slot-indexed pool.
//
// "Inference for linear attention and hybrid architectures", section "Two
// ways to write the same computation": a decode step reads the d_k x d_v
// state once and applies one rank-one update, so the step is bound by the
// state bytes it moves:
//   GLA:  S <- alpha S + k^T v                      o = q S = alpha (q S_old) + (q.k) v
//   GDN:  u = beta (v - alpha (k S_old))            S <- alpha S_old + k^T u
//         o = q S = alpha (q S_old) + (q.k) u
//   NLA:  (normalised linear attention, phi = elu + 1, no gates, normaliser z)
//         S <- S + phi(k)^T v,  z <- z + phi(k),
//         o = phi(q) S / (phi(q) . z + 1e-6) = (phi(q) S_old + (q.k) v) / (phi(q) . z_old + q.k + 1e-6)
// Section "Speculative decoding and PD disaggregation": requests address their
// states by slot, and speculative decode keeps one state per draft position.
//
// Kernel design (sm_103a).  A state's columns evolve independently, so a
// 2-CTA cluster owns a (request, head) unit: CTA `half` holds the 128 x 64
// column half in shared memory.  Clusters are persistent: each walks a
// contiguous range of units (head-major, so the conv weights of a head stay
// in registers) through a two-deep ring.  For every unit one thread issues,
// two units ahead, a TMA tile load of the state half plus bulk copies of the
// unit's conv history and token rows, all completing on the ring slot's
// mbarrier; slot ids, gates and destination slots come from a small table
// filled by 4-byte async copies three units ahead.  While a unit is computed,
// the next one's bytes are already in flight, so the memory system sees a
// steady stream of 32 KiB reads and writes instead of a chain of dependent
// round trips per unit.  Decode and speculative decode run this same code, so
// a draft state equals the state of repeated decode steps bit for bit.
//
// The two halves of a unit read the q / k conv history; half 0 writes it
// back (in place for decode).  Each CTA arrives on the cluster barrier once its
// copy of the unit has landed and waits on it before its first history write.
#include <string.h>

#include "common.cuh"
#include "frontend.cuh"
#include "prefill_tc.cuh"
#include "sm100.cuh"

namespace glinattn {
namespace {

using namespace sm100;

constexpr int kD = 128;               // d_k = d_v
constexpr int kDC = 64;               // state columns per CTA
constexpr int kNT = 128;              // threads per CTA
constexpr int kNW = kNT / 32;
constexpr int kColG = kDC / 4;        // 16-byte column groups
constexpr int kRowG = kNT / kColG;    // 8 row groups
constexpr int kRPT = kD / kRowG;      // 16 rows per thread
constexpr int kNCH = 2 * kD + kDC;    // front-end channels: q, k, own v slice
constexpr int kMaxC = (kNCH + kNT - 1) / kNT;
constexpr int kTab = 4;               // unit table entries
constexpr int kTabSteps = 8;          // per-step scalars kept in a table entry
constexpr int kTabWords = 32;         // [0] src slot, [1..8] dst slots, [9..16] alpha, [17..24] beta,
                                      // [25] steps applied (replay)
constexpr uint32_t kStateBytes = kD * kDC * 4;
// units in flight per CTA (the ring depth): two for decode, whose one step per
// unit is short next to a state's copy; one for several steps per unit, where
// the smaller footprint lets 5 CTAs (20 warps) share an SM to hide the latency
// of each step's reductions
__host__ __device__ constexpr uint32_t misc_bytes(int kr) {
  return kNCH * 4 + kNW * 2 * kDC * 4 + 4 * kNW * 4 + kTab * kTabWords * 4 + kr * 8;
}

// token rows of a unit carried in its ring slot: 2 with two slots (3 CTAs per
// SM), 4 with one (5 CTAs per SM); later rows come from global memory
__host__ __device__ constexpr int ring_steps(int kr) { return kr == 1 ? 4 : 2; }
// ring slot: the state half, then the conv history (3 rows) and the first
// `xrows` token rows of the unit, each row kNCH channels of `esz` bytes
__host__ __device__ constexpr int ring_xrows(int steps, int kr) { return steps < ring_steps(kr) ? steps : ring_steps(kr); }
__host__ __device__ constexpr uint32_t small_bytes(int esz, int xrows) { return (3u + xrows) * kNCH * esz; }
// the state slice, the small rows, then (normalised linear attention only) the
// normaliser z: 512 bytes, a multiple of 128 like the rest
__host__ __device__ constexpr uint32_t slot_bytes(int esz, int xrows, bool nla) {
  return kStateBytes + small_bytes(esz, xrows) + (nla ? kD * 4 : 0);
}
__host__ __device__ constexpr uint32_t smem_bytes(int esz, int xrows, int kr, bool nla) {
  return 128 + kr * slot_bytes(esz, xrows, nla) + misc_bytes(kr);
}

__device__ __forceinline__ void cp_async4(void *dst, const void *src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ float ld_act(const void *base, size_t idx, int bf16) {
  if (bf16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(base)[idx]);
  return reinterpret_cast<const float *>(base)[idx];
}

__device__ __forceinline__ void st_act(void *base, size_t idx, float x, int bf16) {
  if (bf16)
    reinterpret_cast<__nv_bfloat16 *>(base)[idx] = __float2bfloat16_rn(x);
  else
    reinterpret_cast<float *>(base)[idx] = x;
}

// phi(x) = elu(x) + 1, the positive feature map of normalised linear attention
__device__ __forceinline__ float feature_map(float x) { return x > 0.f ? x + 1.f : expf(x); }

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// kNla: normalised linear attention as a template parameter, so the gated
// instances carry none of its code
// kOut: the call writes outputs (a replay does not: then the q S row
// products, the q . k scalars and their reductions are skipped)
template <int kRing, bool kNla, bool kOut>
__global__ void __launch_bounds__(kNT, kRing == 1 ? 5 : 4) decode128_kernel(const __grid_constant__ CUtensorMap tstate,
                                                        const RecurParams p) {
  extern __shared__ uint8_t smem_raw[];
  // 128-byte aligned base derived from the shared array itself, so the compiler
  // keeps every access below in the shared state space
  uint8_t *smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
  const int in_bf16 = p.in_bf16;
  const int esz = in_bf16 ? 2 : 4;
  const int xrows = ring_xrows(p.steps, kRing);
  const uint32_t sbytes = slot_bytes(esz, xrows, kNla);
  float *s_act = reinterpret_cast<float *>(smem + kRing * sbytes);  // q | k | own v slice
  float *s_red = s_act + kNCH;                                      // [warp][k S | q S][kDC]
  float *s_wsum = s_red + kNW * 2 * kDC;                            // [|q|^2, |k|^2, q.k, q.z][warp]
  int *s_tab = reinterpret_cast<int *>(s_wsum + 4 * kNW);           // [kTab][kTabWords]
  uint64_t *s_full = reinterpret_cast<uint64_t *>(s_tab + kTab * kTabWords);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int half = blockIdx.x & 1;
  const int cluster = blockIdx.x >> 1, nclusters = gridDim.x >> 1;
  const int col0 = half * kDC;
  const int cg = tid % kColG, rg = tid / kColG;
  const int H = p.H, N = p.N, steps = p.steps;
  const long long U = (long long)N * H;  // at most 2^30 (checked by the caller)
  const int u0 = (int)(U * cluster / nclusters);
  const int K = (int)(U * (cluster + 1) / nclusters) - u0;
  const bool conv = p.conv_w != nullptr;
  const bool gdn = p.variant == GLINATTN_GDN;
  constexpr bool nla = kNla;  // no gates; phi(q), phi(k); z beside the state
  const int tsteps = steps < kTabSteps ? steps : kTabSteps;
  const int ndst = p.dst_per_step ? steps : 1;
  const size_t DD = (size_t)kD * kD;

  // unit k of this cluster: head-major order, so consecutive units share a head
  auto unit_h = [&](int k) { return (u0 + k) / N; };
  auto unit_n = [&](int k) { return (u0 + k) - ((u0 + k) / N) * N; };
  // global conv channel of local channel c (q, k, own v slice) of head h
  auto chan = [&](int c, int h) {
    if (c < 2 * kD) return (c / kD) * H * kD + h * kD + (c % kD);
    return 2 * H * kD + h * kD + col0 + (c - 2 * kD);
  };

  // ---- per-unit scalars: 4-byte async copies into a table entry (warp 0) -------
  auto tab_issue = [&](int k) {
    if (warp != 0) return;
    if (k < K) {
      const int n = unit_n(k), h = unit_h(k);
      int *e = s_tab + (k % kTab) * kTabWords;
      if (lane == 0) {
        cp_async4(&e[0], &p.src_slot[n]);
      } else if (lane <= kTabSteps) {
        const int t = lane - 1;
        if (t < tsteps && t < ndst && p.dst_slot) cp_async4(&e[lane], &p.dst_slot[(size_t)n * ndst + t]);
      } else if (lane <= 2 * kTabSteps) {
        const int t = lane - 1 - kTabSteps;
        if (t < tsteps && !nla) cp_async4(&e[lane], &p.alpha[((size_t)n * steps + t) * H + h]);
      } else if (lane <= 3 * kTabSteps) {
        const int t = lane - 1 - 2 * kTabSteps;
        if (t < tsteps && gdn) cp_async4(&e[lane], &p.beta[((size_t)n * steps + t) * H + h]);
      } else if (lane == 3 * kTabSteps + 1 && p.step_count) {
        cp_async4(&e[lane], &p.step_count[n]);
      }
    }
    cp_async_commit();  // one group per call, empty past the end
  };

  // ---- ring slot fill: state half, conv history, token row 0 (thread 0) --------
  auto ring_issue = [&](int k) {
    const int *e = s_tab + (k % kTab) * kTabWords;
    uint64_t *bar = &s_full[k % kRing];
    const int slot = e[0];
    const int su = p.step_count ? e[1 + 3 * kTabSteps] : steps;
    if (slot < 0 || slot >= p.pool_slots || su <= 0 || su > steps) {  // nothing to load; reported when
      mbar_arrive(bar);                                              // the unit is computed
      return;
    }
    const int n = unit_n(k), h = unit_h(k);
    uint8_t *st = smem + (k % kRing) * sbytes;
    uint8_t *small = st + kStateBytes;
    const uint32_t bytes = kStateBytes + (conv ? 3u : 0u) * kNCH * esz + (uint32_t)xrows * kNCH * esz +
                           (nla ? kD * 4u : 0u);
    mbar_arrive_expect_tx(bar, bytes);
    tma_load_3d(st, &tstate, bar, col0, 0, slot * H + h);
    if (nla) bulk_load(small + small_bytes(esz, xrows), p.z_src + ((size_t)slot * H + h) * kD, kD * 4, bar);
    if (conv) {
#pragma unroll
      for (int j = 0; j < 3; ++j) {
        const uint8_t *row = (const uint8_t *)p.conv_src + ((size_t)slot * 3 + j) * p.Cch * esz;
        uint8_t *dst = small + (size_t)j * kNCH * esz;
        bulk_load(dst, row + (size_t)(h * kD) * esz, kD * esz, bar);
        bulk_load(dst + kD * esz, row + (size_t)(H * kD + h * kD) * esz, kD * esz, bar);
        bulk_load(dst + 2 * kD * esz, row + (size_t)(2 * H * kD + h * kD + col0) * esz, kDC * esz, bar);
      }
    }
    for (int t = 0; t < xrows; ++t) {
      const size_t row = ((size_t)n * steps + t) * H + h;
      uint8_t *xs = small + (size_t)(3 + t) * kNCH * esz;
      bulk_load(xs, (const uint8_t *)p.q + row * kD * esz, kD * esz, bar);
      bulk_load(xs + kD * esz, (const uint8_t *)p.k + row * kD * esz, kD * esz, bar);
      bulk_load(xs + 2 * kD * esz, (const uint8_t *)p.v + (row * kD + col0) * esz, kDC * esz, bar);
    }
  };

  if (tid == 0) {
    for (int s = 0; s < kRing; ++s) mbar_init(&s_full[s], 1);
    fence_mbar_init();
    prefetch_tensormap(&tstate);
  }
  tab_issue(0);
  tab_issue(1);
  tab_issue(2);
  if (warp == 0) cp_async_wait<1>();
  __syncthreads();
  int issued = 0, landed = 0;  // ring units issued / seen complete (thread 0's count)
  if (tid == 0) {
    for (int k = 0; k < kRing && k < K; ++k) ring_issue(k);
    issued = K < kRing ? K : kRing;
  }

  float wr[kMaxC][4], wn[kMaxC][4];  // conv weights of the current / next head
  int h_w = -1, h_wn = -1;
  auto load_w = [&](float (&w)[kMaxC][4], int h) {
#pragma unroll
    for (int i = 0; i < kMaxC; ++i) {
      const int c = tid + i * kNT;
      w[i][0] = w[i][1] = w[i][2] = 0.f;
      w[i][3] = 1.f;
      if (conv && c < kNCH) {
        const float4 v4 = *reinterpret_cast<const float4 *>(p.conv_w + (size_t)chan(c, h) * 4);
        w[i][0] = v4.x; w[i][1] = v4.y; w[i][2] = v4.z; w[i][3] = v4.w;
      }
    }
  };
  if (K > 0) {
    load_w(wr, unit_h(0));
    h_w = unit_h(0);
  }

  bool dead = false;  // a ring wait timed out: no further copies or compute
  for (int k = 0; k < K; ++k) {
    const int s = k % kRing;
    const int n = unit_n(k), h = unit_h(k);
    tab_issue(k + 3);
    if (h != h_w) {  // head change: take the prefetched weights (or load them)
      if (h == h_wn) {
#pragma unroll
        for (int i = 0; i < kMaxC; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) wr[i][j] = wn[i][j];
      } else {
        load_w(wr, h);
      }
      h_w = h;
    }
    if (k + 1 < K && unit_h(k + 1) != h && unit_h(k + 1) != h_wn) {
      load_w(wn, unit_h(k + 1));
      h_wn = unit_h(k + 1);
    }

    bool ok = true;
    if (!dead) {
      ok = mbar_wait(&s_full[s], (uint32_t)(k / kRing) & 1u);
      if (ok) landed = k + 1;
    }
    cluster_arrive_relaxed();  // this CTA's copy of the unit's conv history has landed

    // ---- validation from the table (uniform): slots in range, gates in (0, 1] ----
    const int *e = s_tab + (k % kTab) * kTabWords;
    int bad = 0;
    // steps applied to this unit: all, or the request's accepted length (replay)
    int su = steps;
    if (!dead && p.step_count) {
      su = e[1 + 3 * kTabSteps];
      if (su < 0 || su > steps) {
        bad |= GLINATTN_DEV_BAD_COUNT;
        su = 0;
      }
    }
    if (!dead) {
      const int slot = e[0];
      if (slot < 0 || slot >= p.pool_slots) bad |= GLINATTN_DEV_BAD_SLOT;
      for (int t = 0; t < tsteps && t < ndst && p.dst_slot; ++t) {
        const int d = e[1 + t];
        if (d < 0 || d >= p.pool_slots) bad |= GLINATTN_DEV_BAD_SLOT;
      }
      for (int t = 0; t < tsteps && t < su && !nla; ++t) {
        const float a = __int_as_float(e[1 + kTabSteps + t]);
        if (!(a > 0.f && a <= 1.f)) bad |= GLINATTN_DEV_BAD_GATE;
      }
      if (steps > kTabSteps) {  // the steps beyond the table, checked in global memory
        int b2 = 0;
        for (int t = kTabSteps + tid; t < steps; t += kNT) {
          const float a = nla ? 1.f : p.alpha[((size_t)n * steps + t) * H + h];
          if (t < su && !(a > 0.f && a <= 1.f)) b2 |= GLINATTN_DEV_BAD_GATE;
          if (t < ndst && p.dst_slot) {
            const int d = p.dst_slot[(size_t)n * ndst + t];
            if (d < 0 || d >= p.pool_slots) b2 |= GLINATTN_DEV_BAD_SLOT;
          }
        }
        if (__syncthreads_or(b2 & GLINATTN_DEV_BAD_SLOT)) bad |= GLINATTN_DEV_BAD_SLOT;
        if (__syncthreads_or(b2 & GLINATTN_DEV_BAD_GATE)) bad |= GLINATTN_DEV_BAD_GATE;
      }
      if (bad && half == 0 && tid == 0 && p.dev_status) atomicOr(p.dev_status, (uint32_t)bad);
    }
    bool hist_waited = false;

    if (!dead && !bad && su > 0) {
      float *sst = reinterpret_cast<float *>(smem + s * sbytes);
      float4 *st4 = reinterpret_cast<float4 *>(sst);
      const uint8_t *small = smem + s * sbytes + kStateBytes;
      float *zs = reinterpret_cast<float *>(smem + s * sbytes + kStateBytes + small_bytes(esz, xrows));  // z (NLA)
      // raw input of local channel c at step st: the ring slot's rows for the
      // first xrows steps, global memory after that
      auto x_at = [&](int st, int c) -> float {
        if (st < xrows) return ld_act(small, (3 + st) * kNCH + c, in_bf16);
        const void *src = c < kD ? p.q : (c < 2 * kD ? p.k : p.v);
        const int ci = c < 2 * kD ? (c % kD) : col0 + (c - 2 * kD);
        return ld_act(src, (((size_t)n * steps + st) * H + h) * kD + ci, in_bf16);
      };
      // inputs of this step (xr) and of the next two (xa, xb): global loads are
      // issued two steps before their use
      float xr[kMaxC], xa[kMaxC], xb[kMaxC], hr[kMaxC][3];
#pragma unroll
      for (int i = 0; i < kMaxC; ++i) {
        const int c = tid + i * kNT;
        xr[i] = xa[i] = xb[i] = 0.f;
        hr[i][0] = hr[i][1] = hr[i][2] = 0.f;
        if (c < kNCH) {
          xr[i] = x_at(0, c);
          if (su > 1) xa[i] = x_at(1, c);
          if (su > 2) xb[i] = x_at(2, c);
          if (conv)
#pragma unroll
            for (int j = 0; j < 3; ++j) hr[i][j] = ld_act(small, j * kNCH + c, in_bf16);
        }
      }
      float a_nx = nla ? 1.f : __int_as_float(e[1 + kTabSteps]);
      float b_nx = gdn ? __int_as_float(e[1 + 2 * kTabSteps]) : 0.f;
      int d_nx = e[1];

      for (int t = 0; t < su; ++t) {
        const size_t row = ((size_t)n * steps + t) * H + h;  // (n, t, h)
        const float a = a_nx, bgate = b_nx;
        const int dslot = d_nx;
        const bool last = t == su - 1;
        const bool emit = p.S_dst && (p.dst_per_step || last);
        if (!last) {  // next step's scalars: table, else global memory
          const int t1 = t + 1;
          if (t1 < kTabSteps) {
            a_nx = nla ? 1.f : __int_as_float(e[1 + kTabSteps + t1]);
            if (gdn) b_nx = __int_as_float(e[1 + 2 * kTabSteps + t1]);
            if (p.dst_per_step) d_nx = e[1 + t1];
          } else {
            a_nx = nla ? 1.f : p.alpha[row + H];
            if (gdn) b_nx = p.beta[row + H];
            if (p.dst_per_step && p.dst_slot) d_nx = p.dst_slot[(size_t)n * ndst + t1];
          }
        }
        // ---- front end: conv, history shift, next token prefetch, L2 norms ------
        float yv[kMaxC];
        float sq = 0.f, sk = 0.f;
#pragma unroll
        for (int i = 0; i < kMaxC; ++i) {
          const int c = tid + i * kNT;
          const float x = xr[i];
          // without outputs q' is not needed (i = 0 holds the q channels)
          float y = 0.f;
          if (kOut || i > 0) {
            y = conv ? fe::conv4(wr[i][0], wr[i][1], wr[i][2], wr[i][3], hr[i][0], hr[i][1], hr[i][2], x) : x;
            if (nla && c < 2 * kD) y = feature_map(y);
          }
          yv[i] = y;
          // one q and one k channel per thread (channel tid of each)
          if (c < kD) {
            if (kOut) sq = __fmul_rn(y, y);
          } else if (c < 2 * kD) {
            sk = __fmul_rn(y, y);
          }
          hr[i][0] = hr[i][1];
          hr[i][1] = hr[i][2];
          hr[i][2] = x;
          if (c < kNCH && !last) {  // shift the input queue; step t + 3 is loaded now
            xr[i] = xa[i];
            xa[i] = xb[i];
            if (t + 3 < su) xb[i] = x_at(t + 3, c);
          }
        }
        float iq = 1.f, ik = 1.f;
        if (p.qk_l2norm) {  // pairwise sums of squares: lanes, then warps
          if (kOut) sq = fe::warp_pairwise_sum(sq);
          sk = fe::warp_pairwise_sum(sk);
          if (lane == 0) {
            if (kOut) s_wsum[warp] = sq;
            s_wsum[kNW + warp] = sk;
          }
          __syncthreads();
          if (kOut) iq = fe::inv_norm(fe::pairwise_sum<kNW>(s_wsum));
          ik = fe::inv_norm(fe::pairwise_sum<kNW>(s_wsum + kNW));
        }
        const bool round_act = in_bf16 && (conv || p.qk_l2norm || nla);
        float qk_part = 0.f, qz_part = 0.f;
        {
          float qv = 0.f;
#pragma unroll
          for (int i = 0; i < kMaxC; ++i) {
            const int c = tid + i * kNT;
            if (c < kNCH) {
              float y = yv[i];
              if (c < kD) y = __fmul_rn(y, iq);
              else if (c < 2 * kD) y = __fmul_rn(y, ik);
              if (round_act) y = __bfloat162float(__float2bfloat16_rn(y));
              s_act[c] = y;
              if (c < kD) {
                qv = y;
                if (nla) qz_part = y * zs[c];
              } else if (c < 2 * kD) {
                qk_part = qv * y;  // q_c * k_c: same thread, same c % kD
              }
            }
          }
        }
        if (kOut) {
          qk_part = warp_sum(qk_part);
          if (lane == 0) s_wsum[2 * kNW + warp] = qk_part;
          if (nla) {
            qz_part = warp_sum(qz_part);
            if (lane == 0) s_wsum[3 * kNW + warp] = qz_part;
          }
        }
        if (!__syncthreads_and(ok)) {
          dead = true;
          break;
        }
        float qk = 0.f, qz = 0.f;
        if (kOut) {
#pragma unroll
          for (int w = 0; w < kNW; ++w) qk += s_wsum[2 * kNW + w];
        }
        if (nla) {
          if (kOut) {
#pragma unroll
            for (int w = 0; w < kNW; ++w) qz += s_wsum[3 * kNW + w];
          }
          // z <- z + phi(k): channel tid, read above only by this thread
          zs[tid] += s_act[kD + tid];
        }

        // ---- partial k S and q S over this thread's rows, then across rows ------
        const float *sqa = s_act, *ska = s_act + kD, *sva = s_act + 2 * kD;
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f), y = x;
#pragma unroll
        for (int i = 0; i < kRPT; ++i) {
          const int r = rg + kRowG * i;
          const float4 S = st4[r * kColG + cg];
          const float kr = ska[r], qr = sqa[r];
          x.x += kr * S.x; x.y += kr * S.y; x.z += kr * S.z; x.w += kr * S.w;
          if (kOut) {
            y.x += qr * S.x; y.y += qr * S.y; y.z += qr * S.z; y.w += qr * S.w;
          }
        }
        // the warp's two row groups (lanes l and l ^ 16 share a column group)
        x.x += __shfl_xor_sync(0xffffffffu, x.x, 16);
        x.y += __shfl_xor_sync(0xffffffffu, x.y, 16);
        x.z += __shfl_xor_sync(0xffffffffu, x.z, 16);
        x.w += __shfl_xor_sync(0xffffffffu, x.w, 16);
        if (kOut) {
          y.x += __shfl_xor_sync(0xffffffffu, y.x, 16);
          y.y += __shfl_xor_sync(0xffffffffu, y.y, 16);
          y.z += __shfl_xor_sync(0xffffffffu, y.z, 16);
          y.w += __shfl_xor_sync(0xffffffffu, y.w, 16);
        }
        if (lane < 16) {
          *reinterpret_cast<float4 *>(&s_red[(warp * 2 + 0) * kDC + 4 * cg]) = x;
          if (kOut) *reinterpret_cast<float4 *>(&s_red[(warp * 2 + 1) * kDC + 4 * cg]) = y;
        }
        __syncthreads();
        x = make_float4(0.f, 0.f, 0.f, 0.f);
        y = x;
#pragma unroll
        for (int w = 0; w < kNW; ++w) {
          const float4 a4 = *reinterpret_cast<const float4 *>(&s_red[(w * 2 + 0) * kDC + 4 * cg]);
          const float4 b4 = kOut ? *reinterpret_cast<const float4 *>(&s_red[(w * 2 + 1) * kDC + 4 * cg]) : a4;
          x.x += a4.x; x.y += a4.y; x.z += a4.z; x.w += a4.w;
          if (kOut) {
            y.x += b4.x; y.y += b4.y; y.z += b4.z; y.w += b4.w;
          }
        }

        // ---- update: shared copy for the next step, global copy when due --------
        const float4 vv = *reinterpret_cast<const float4 *>(sva + 4 * cg);
        float4 u = vv;
        if (gdn) {
          u.x = bgate * (vv.x - a * x.x);
          u.y = bgate * (vv.y - a * x.y);
          u.z = bgate * (vv.z - a * x.z);
          u.w = bgate * (vv.w - a * x.w);
        }
        float *dst = emit ? p.S_dst + ((size_t)dslot * H + h) * DD + col0 : nullptr;
#pragma unroll
        for (int i = 0; i < kRPT; ++i) {
          const int r = rg + kRowG * i;
          const float kr = ska[r];
          float4 S = st4[r * kColG + cg];
          S.x = a * S.x + kr * u.x;
          S.y = a * S.y + kr * u.y;
          S.z = a * S.z + kr * u.z;
          S.w = a * S.w + kr * u.w;
          if (!last) st4[r * kColG + cg] = S;
          if (emit) *reinterpret_cast<float4 *>(dst + (size_t)r * kD + 4 * cg) = S;
        }
        if (kOut && rg == 0 && p.o) {
          // normalised linear attention divides by phi(q) . z_{t-1} + phi(q) . phi(k) + eps
          const float inv = nla ? 1.f / (qz + qk + 1e-6f) : 1.f;
          const float o0 = (a * y.x + qk * u.x) * inv, o1 = (a * y.y + qk * u.y) * inv;
          const float o2 = (a * y.z + qk * u.z) * inv, o3 = (a * y.w + qk * u.w) * inv;
          const size_t ob = row * kD + col0 + 4 * cg;
          if (p.out_bf16) {
            const __nv_bfloat162 lo = __floats2bfloat162_rn(o0, o1), hi = __floats2bfloat162_rn(o2, o3);
            uint2 pk;
            pk.x = *reinterpret_cast<const uint32_t *>(&lo);
            pk.y = *reinterpret_cast<const uint32_t *>(&hi);
            *reinterpret_cast<uint2 *>(reinterpret_cast<__nv_bfloat16 *>(p.o) + ob) = pk;
          } else {
            *reinterpret_cast<float4 *>(reinterpret_cast<float *>(p.o) + ob) = make_float4(o0, o1, o2, o3);
          }
        }
        if (emit && nla && half == 0 && p.z_dst) {  // z after this step (the other half has its copy)
          if (!hist_waited) {
            cluster_wait();
            hist_waited = true;
          }
          p.z_dst[((size_t)dslot * H + h) * kD + tid] = zs[tid];
        }
        if (emit && conv && p.conv_dst) {
          if (!hist_waited) {
            cluster_wait();
            hist_waited = true;
          }
#pragma unroll
          for (int i = 0; i < kMaxC; ++i) {
            const int c = tid + i * kNT;
            if (c < kNCH && (c >= 2 * kD || half == 0))
#pragma unroll
              for (int j = 0; j < 3; ++j)
                st_act(p.conv_dst, ((size_t)dslot * 3 + j) * p.Cch + chan(c, h), hr[i][j], in_bf16);
          }
        }
        if (!last) __syncthreads();  // the next step overwrites s_act and s_red
      }
    }
    if (!hist_waited) cluster_wait();

    // ---- end of unit: the ring slot is free, the table entry two ahead is ready ---
    if (warp == 0) cp_async_wait<1>();
    if (!__syncthreads_and(ok)) dead = true;
    if (tid == 0 && !dead && k + kRing < K) {
      ring_issue(k + kRing);
      issued = k + kRing + 1;
    }
  }

  // copies still in flight (only after a timeout) land before the CTA exits
  if (tid == 0) {
    for (int k = landed; k < issued; ++k) mbar_wait(&s_full[k % kRing], (uint32_t)(k / kRing) & 1u);
    if (dead && p.dev_status) atomicOr(p.dev_status, GLINATTN_DEV_WAIT_TIMEOUT);
  }
  if (warp == 0) cp_async_wait<0>();
}

}  // namespace

bool decode128_supports(const RecurParams &p, int d) {
  return d == kD && p.src_slot != nullptr && (p.dst_slot != nullptr || p.S_dst == nullptr) && p.S_src != nullptr &&
         p.steps >= 1 && p.pool_slots > 0 && (p.conv_w == nullptr || p.conv_src != nullptr) &&
         p.S_blocks == nullptr && p.Hq == p.H &&
         (p.variant != GLINATTN_NLA ||  // the normaliser pool is copied in with the state
          (p.z_src != nullptr && ((uintptr_t)p.z_src & 15u) == 0 && ((uintptr_t)p.z_dst & 15u) == 0));
}

template <int kRing, bool kNla, bool kOut>
cudaError_t launch_ring(const RecurParams &p, cudaStream_t stream) {
  const int esz = p.in_bf16 ? 2 : 4;
  const int smem = (int)smem_bytes(esz, ring_xrows(p.steps, kRing), kRing, kNla);
  CUtensorMap tmap;
  memset(&tmap, 0, sizeof(tmap));
  {
    // the pool as (columns, rows, slot * H + head) planes; box = one column half
    const long long dims[3] = {kD, kD, (long long)p.pool_slots * p.H};
    const int box[3] = {kDC, kD, 1};
    if (!encode_3d_map(&tmap, p.S_src, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, dims, box, false))
      return cudaErrorInvalidValue;
  }
  cudaError_t e = cudaFuncSetAttribute(decode128_kernel<kRing, kNla, kOut>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(decode128_kernel<kRing, kNla, kOut>, cudaFuncAttributePreferredSharedMemoryCarveout,
                           (int)cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kNT);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;  // the two column halves of a state
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // as many clusters as fit on the GPU at once, never more than there are units
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  int max_clusters = 0;
  cfg.gridDim = dim3(2 * (unsigned)sms);
  if ((e = cudaOccupancyMaxActiveClusters(&max_clusters, decode128_kernel<kRing, kNla, kOut>, &cfg)) != cudaSuccess) return e;
  if (max_clusters < 1) max_clusters = 1;
  const long long units = (long long)p.N * p.H;
  const long long clusters = units < max_clusters ? units : max_clusters;
  cfg.gridDim = dim3((unsigned)(2 * clusters));
  return cudaLaunchKernelEx(&cfg, decode128_kernel<kRing, kNla, kOut>, tmap, p);
}

template <bool kOut>
cudaError_t launch_decode128_out(const RecurParams &p, cudaStream_t stream) {
  if (p.variant == GLINATTN_NLA)
    return p.steps > 1 ? launch_ring<1, true, kOut>(p, stream) : launch_ring<2, true, kOut>(p, stream);
  return p.steps > 1 ? launch_ring<1, false, kOut>(p, stream) : launch_ring<2, false, kOut>(p, stream);
}

cudaError_t launch_decode128(const RecurParams &p, cudaStream_t stream) {
  return p.o ? launch_decode128_out<true>(p, stream) : launch_decode128_out<false>(p, stream);
}

}  // namespace glinattn
