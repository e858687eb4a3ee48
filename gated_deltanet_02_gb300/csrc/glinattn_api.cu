// glinattn_api.cu -- the extern "C" boundary: host-side argument validation
// and dispatch to the kernels.  Nothing is launched when validation fails.
#include <stdio.h>
#include <stdlib.h>

#include "common.cuh"
#include "prefill_tc.cuh"

namespace {

using glinattn::RecurParams;

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

bool supported_head(int d) { return d == 16 || d == 32 || d == 64 || d == 128; }

// [a, a+na) and [b, b+nb) overlap without being the same buffer
bool partial_overlap(const void *a, size_t na, const void *b, size_t nb) {
  if (!a || !b || a == b) return false;
  const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
  return x < y + nb && y < x + na;
}

glinattn_status check_common(int variant, int in_dtype, int out_dtype, int dk, int dv,
                             int heads) {
  if (variant != GLINATTN_GLA && variant != GLINATTN_GDN && variant != GLINATTN_NLA)
    return GLINATTN_ERR_INVALID_ARG;
  if ((in_dtype != GLINATTN_F32 && in_dtype != GLINATTN_BF16) ||
      (out_dtype != GLINATTN_F32 && out_dtype != GLINATTN_BF16))
    return GLINATTN_ERR_INVALID_ARG;
  if (heads <= 0 || dk <= 0 || dv <= 0) return GLINATTN_ERR_INVALID_ARG;
  // square heads, or the 128 x 64 state of the SSD form (state 128, head dim 64)
  const bool shape_ok = (dk == dv && supported_head(dk)) || (dk == 128 && dv == 64);
  if (!shape_ok) return GLINATTN_ERR_UNSUPPORTED;
  return GLINATTN_OK;
}

// q / k heads: 0 means one per head; otherwise a divisor of heads (groups of
// heads share q and k).  Grouped heads take no convolution.
glinattn_status check_qk_heads(int qk_heads, int heads, bool conv, int *out) {
  const int hq = qk_heads == 0 ? heads : qk_heads;
  if (hq < 0 || hq > heads || heads % hq != 0) return GLINATTN_ERR_INVALID_ARG;
  if (hq != heads && conv) return GLINATTN_ERR_UNSUPPORTED;
  *out = hq;
  return GLINATTN_OK;
}

template <typename... P>
bool all_aligned(P... ptrs) {
  const void *list[] = {ptrs...};
  for (const void *p : list)
    if (p && !aligned16(p)) return false;
  return true;
}

}  // namespace

extern "C" {

const char *glinattn_status_string(glinattn_status s) {
  switch (s) {
    case GLINATTN_OK: return "ok";
    case GLINATTN_ERR_INVALID_ARG: return "invalid argument";
    case GLINATTN_ERR_UNSUPPORTED: return "unsupported configuration";
    case GLINATTN_ERR_CUDA: return "CUDA error";
    case GLINATTN_ERR_DEVICE_STATUS: return "device reported an error status";
    case GLINATTN_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

int glinattn_version(void) { return 100; /* 0.1.0 */ }

size_t glinattn_state_bytes(int heads, int dk, int dv) {
  if (heads <= 0 || dk <= 0 || dv <= 0) return 0;
  return (size_t)heads * dk * dv * sizeof(float);
}

glinattn_status glinattn_prefill(const glinattn_prefill_args *a, glinattn_stream_t stream) {
  if (!a) return GLINATTN_ERR_INVALID_ARG;
  glinattn_status st = check_common(a->variant, a->in_dtype, a->out_dtype, a->dk, a->dv, a->heads);
  if (st != GLINATTN_OK) return st;
  if (a->batch < 0 || a->seqlen < 0) return GLINATTN_ERR_INVALID_ARG;
  const int B = a->batch, T = a->seqlen, H = a->heads, dk = a->dk, dv = a->dv;
  int Hq = H;
  st = check_qk_heads(a->qk_heads, H, a->conv_w != nullptr, &Hq);
  if (st != GLINATTN_OK) return st;
  if ((long long)B * H > (1ll << 30) || (long long)T > (1ll << 30)) return GLINATTN_ERR_INVALID_ARG;
  if (B == 0) return GLINATTN_OK;
  const size_t act = a->in_dtype == GLINATTN_BF16 ? 2 : 4;
  const size_t state_bytes = (size_t)B * H * dk * dv * sizeof(float);
  if (!a->S_T) return GLINATTN_ERR_INVALID_ARG;
  if (a->state_every < 0) return GLINATTN_ERR_INVALID_ARG;
  const bool nla = a->variant == GLINATTN_NLA;
  if (nla) {  // no convolution, L2 norm or checkpoints; the normaliser goes out
    if (a->conv_w || a->qk_l2norm || a->state_every) return GLINATTN_ERR_UNSUPPORTED;
    if (!a->z_T) return GLINATTN_ERR_INVALID_ARG;
  }
  const bool emit_blocks = a->state_every > 0 && T / a->state_every > 0;
  if (emit_blocks && (!a->S_blocks || !aligned16(a->S_blocks))) return GLINATTN_ERR_INVALID_ARG;
  if (T > 0) {
    if (!a->q || !a->k || !a->v || (!a->alpha && !nla) || !a->o) return GLINATTN_ERR_INVALID_ARG;
    if (a->variant == GLINATTN_GDN && !a->beta) return GLINATTN_ERR_INVALID_ARG;
  }
  if (!all_aligned(a->q, a->k, a->v, a->alpha, a->beta, a->S0, a->S_T, a->o, a->conv_w,
                   a->conv_in, a->conv_out))
    return GLINATTN_ERR_INVALID_ARG;
  if (nla && !all_aligned(a->z0, a->z_T)) return GLINATTN_ERR_INVALID_ARG;
  if (partial_overlap(a->S0, state_bytes, a->S_T, state_bytes)) return GLINATTN_ERR_INVALID_ARG;
  if (nla && partial_overlap(a->z0, (size_t)B * H * dk * 4, a->z_T, (size_t)B * H * dk * 4))
    return GLINATTN_ERR_INVALID_ARG;
  const int Cch = H * (2 * dk + dv);
  if (a->conv_w) {
    const size_t cb = (size_t)B * 3 * Cch * act;
    if (partial_overlap(a->conv_in, cb, a->conv_out, cb)) return GLINATTN_ERR_INVALID_ARG;
  }

  // the chunked kernels emit states at chunk ends only (checked whatever the device)
  if ((glinattn::prefill_tc_supports(*a) || glinattn::gdn_tc_supports(*a)) && emit_blocks &&
      a->state_every % 64 != 0)
    return GLINATTN_ERR_UNSUPPORTED;
  const bool tc_device = glinattn::prefill_tc_available();
  if (tc_device && glinattn::gdn_tc_supports(*a) &&
      (!a->workspace || a->workspace_bytes < glinattn::gdn_tc_workspace_bytes(*a) || !aligned16(a->workspace)))
    return GLINATTN_ERR_INVALID_ARG;
  if (tc_device && glinattn::nla_tc_supports(*a) &&
      (!a->workspace || a->workspace_bytes < glinattn::nla_tc_workspace_bytes(*a) || !aligned16(a->workspace)))
    return GLINATTN_ERR_INVALID_ARG;
  // conv caches at the block boundaries: taken before the layer runs, since
  // conv_out may alias conv_in
  const bool conv_blocks = a->conv_w && a->conv_blocks && emit_blocks;
  if (conv_blocks) {
    if (!aligned16(a->conv_blocks)) return GLINATTN_ERR_INVALID_ARG;
    const glinattn_status st = glinattn::launch_conv_blocks(*a, (cudaStream_t)stream);
    if (st != GLINATTN_OK) return st;
  }
  if (tc_device) {
    if (glinattn::prefill_tc_supports(*a)) {
      // few (batch, head) units: split the sequence when the caller gave the scratch for it
      const size_t split = glinattn::gla_split_workspace_bytes(*a);
      if (split && a->workspace && a->workspace_bytes >= split && aligned16(a->workspace))
        return glinattn::launch_gla_split(*a, (cudaStream_t)stream);
      return glinattn::launch_prefill_tc(*a, (cudaStream_t)stream);
    }
    if (glinattn::gdn_tc_supports(*a)) return glinattn::launch_gdn_tc(*a, (cudaStream_t)stream);
    if (glinattn::nla_tc_supports(*a)) return glinattn::launch_nla_tc(*a, (cudaStream_t)stream);
  }

  RecurParams p = {};
  p.variant = a->variant;
  p.in_bf16 = a->in_dtype == GLINATTN_BF16;
  p.out_bf16 = a->out_dtype == GLINATTN_BF16;
  p.qk_l2norm = a->qk_l2norm != 0;
  p.N = B;
  p.steps = T;
  p.H = H;
  p.Hq = Hq;
  p.pool_slots = 0;
  p.Cch = Cch;
  p.q = a->q;
  p.k = a->k;
  p.v = a->v;
  p.alpha = nla ? nullptr : a->alpha;
  p.beta = a->beta;
  p.S_src = a->S0;
  p.S_dst = a->S_T;
  p.z_src = nla ? a->z0 : nullptr;
  p.z_dst = nla ? a->z_T : nullptr;
  p.o = a->o;
  p.conv_w = a->conv_w;
  p.conv_src = a->conv_w ? a->conv_in : nullptr;
  p.conv_dst = a->conv_w ? a->conv_out : nullptr;
  p.dev_status = a->dev_status;
  if (emit_blocks) {
    p.S_blocks = a->S_blocks;
    p.state_every = a->state_every;
    p.nblocks = T / a->state_every;
  }
  return glinattn::launch_recurrent(p, dk, dv, (cudaStream_t)stream);
}

size_t glinattn_prefill_workspace_size(const glinattn_prefill_args *a) {
  if (!a || a->batch <= 0 || a->seqlen <= 0 || a->heads <= 0) return 0;
  if (check_common(a->variant, a->in_dtype, a->out_dtype, a->dk, a->dv, a->heads) != GLINATTN_OK) return 0;
  if (glinattn::nla_tc_supports(*a)) return glinattn::nla_tc_workspace_bytes(*a);
  if (glinattn::prefill_tc_supports(*a)) return glinattn::gla_split_workspace_bytes(*a);
  if (!glinattn::gdn_tc_supports(*a)) return 0;
  return glinattn::gdn_tc_workspace_bytes(*a);
}

glinattn_status glinattn_decode(const glinattn_decode_args *a, glinattn_stream_t stream) {
  if (!a) return GLINATTN_ERR_INVALID_ARG;
  glinattn_status st = check_common(a->variant, a->in_dtype, a->out_dtype, a->dk, a->dv, a->heads);
  if (st != GLINATTN_OK) return st;
  int Hq = a->heads;
  st = check_qk_heads(a->qk_heads, a->heads, a->conv_w != nullptr, &Hq);
  if (st != GLINATTN_OK) return st;
  if (a->num_req < 0 || a->pool_slots <= 0) return GLINATTN_ERR_INVALID_ARG;
  if ((long long)a->num_req * a->heads > (1ll << 30)) return GLINATTN_ERR_INVALID_ARG;
  if (a->num_req == 0) return GLINATTN_OK;
  const bool nla = a->variant == GLINATTN_NLA;
  if (nla && (a->conv_w || a->qk_l2norm)) return GLINATTN_ERR_UNSUPPORTED;
  if (nla && (!a->z_pool || !aligned16(a->z_pool))) return GLINATTN_ERR_INVALID_ARG;
  if (!a->q || !a->k || !a->v || (!a->alpha && !nla) || !a->o || !a->state_pool || !a->slot_ids)
    return GLINATTN_ERR_INVALID_ARG;
  if (a->variant == GLINATTN_GDN && !a->beta) return GLINATTN_ERR_INVALID_ARG;
  if (a->conv_w && !a->conv_pool) return GLINATTN_ERR_INVALID_ARG;
  if (!all_aligned(a->q, a->k, a->v, a->alpha, a->beta, a->state_pool, a->o, a->conv_w, a->conv_pool))
    return GLINATTN_ERR_INVALID_ARG;
  RecurParams p = {};
  p.variant = a->variant;
  p.in_bf16 = a->in_dtype == GLINATTN_BF16;
  p.out_bf16 = a->out_dtype == GLINATTN_BF16;
  p.qk_l2norm = a->qk_l2norm != 0;
  p.N = a->num_req;
  p.steps = 1;
  p.H = a->heads;
  p.Hq = Hq;
  p.pool_slots = a->pool_slots;
  p.Cch = a->heads * (2 * a->dk + a->dv);
  p.q = a->q;
  p.k = a->k;
  p.v = a->v;
  p.alpha = nla ? nullptr : a->alpha;
  p.beta = a->beta;
  p.S_src = a->state_pool;
  p.z_src = nla ? a->z_pool : nullptr;
  p.z_dst = nla ? a->z_pool : nullptr;
  p.src_slot = a->slot_ids;
  p.S_dst = a->state_pool;
  p.dst_slot = a->slot_ids;
  p.dst_per_step = 0;
  p.o = a->o;
  p.conv_w = a->conv_w;
  p.conv_src = a->conv_w ? a->conv_pool : nullptr;
  p.conv_dst = a->conv_w ? a->conv_pool : nullptr;
  p.dev_status = a->dev_status;
  return glinattn::launch_recurrent(p, a->dk, a->dv, (cudaStream_t)stream);
}

glinattn_status glinattn_spec_decode(const glinattn_spec_args *a, glinattn_stream_t stream) {
  if (!a) return GLINATTN_ERR_INVALID_ARG;
  glinattn_status st = check_common(a->variant, a->in_dtype, a->out_dtype, a->dk, a->dv, a->heads);
  if (st != GLINATTN_OK) return st;
  int Hq = a->heads;
  st = check_qk_heads(a->qk_heads, a->heads, a->conv_w != nullptr, &Hq);
  if (st != GLINATTN_OK) return st;
  if (a->num_req < 0 || a->draft_len <= 0 || a->pool_slots <= 0) return GLINATTN_ERR_INVALID_ARG;
  if ((long long)a->num_req * a->heads > (1ll << 30) || a->draft_len > (1 << 20))
    return GLINATTN_ERR_INVALID_ARG;
  if (a->num_req == 0) return GLINATTN_OK;
  const bool nla = a->variant == GLINATTN_NLA;
  if (nla && (a->conv_w || a->qk_l2norm)) return GLINATTN_ERR_UNSUPPORTED;
  if (nla && (!a->z_pool || !aligned16(a->z_pool))) return GLINATTN_ERR_INVALID_ARG;
  if (!a->q || !a->k || !a->v || (!a->alpha && !nla) || !a->o || !a->state_pool || !a->src_slots)
    return GLINATTN_ERR_INVALID_ARG;
  if (a->variant == GLINATTN_GDN && !a->beta) return GLINATTN_ERR_INVALID_ARG;
  if (a->conv_w && !a->conv_pool) return GLINATTN_ERR_INVALID_ARG;
  if (!all_aligned(a->q, a->k, a->v, a->alpha, a->beta, a->state_pool, a->o, a->conv_w, a->conv_pool))
    return GLINATTN_ERR_INVALID_ARG;
  RecurParams p = {};
  p.variant = a->variant;
  p.in_bf16 = a->in_dtype == GLINATTN_BF16;
  p.out_bf16 = a->out_dtype == GLINATTN_BF16;
  p.qk_l2norm = a->qk_l2norm != 0;
  p.N = a->num_req;
  p.steps = a->draft_len;
  p.H = a->heads;
  p.Hq = Hq;
  p.pool_slots = a->pool_slots;
  p.Cch = a->heads * (2 * a->dk + a->dv);
  p.q = a->q;
  p.k = a->k;
  p.v = a->v;
  p.alpha = nla ? nullptr : a->alpha;
  p.beta = a->beta;
  p.S_src = a->state_pool;
  p.z_src = nla ? a->z_pool : nullptr;
  p.z_dst = nla ? a->z_pool : nullptr;
  p.src_slot = a->src_slots;
  const bool verify_only = a->dst_slots == nullptr;  // outputs only, the pool is not written
  p.S_dst = verify_only ? nullptr : a->state_pool;
  p.dst_slot = a->dst_slots;
  p.dst_per_step = verify_only ? 0 : 1;
  p.o = a->o;
  p.conv_w = a->conv_w;
  p.conv_src = a->conv_w ? a->conv_pool : nullptr;
  p.conv_dst = a->conv_w && !verify_only ? a->conv_pool : nullptr;
  p.dev_status = a->dev_status;
  return glinattn::launch_recurrent(p, a->dk, a->dv, (cudaStream_t)stream);
}

glinattn_status glinattn_replay(const glinattn_replay_args *a, glinattn_stream_t stream) {
  if (!a) return GLINATTN_ERR_INVALID_ARG;
  glinattn_status st = check_common(a->variant, a->in_dtype, GLINATTN_F32, a->dk, a->dv, a->heads);
  if (st != GLINATTN_OK) return st;
  int Hq = a->heads;
  st = check_qk_heads(a->qk_heads, a->heads, a->conv_w != nullptr, &Hq);
  if (st != GLINATTN_OK) return st;
  if (a->num_req < 0 || a->draft_len <= 0 || a->pool_slots <= 0) return GLINATTN_ERR_INVALID_ARG;
  if ((long long)a->num_req * a->heads > (1ll << 30) || a->draft_len > (1 << 20))
    return GLINATTN_ERR_INVALID_ARG;
  if (a->num_req == 0) return GLINATTN_OK;
  const bool nla = a->variant == GLINATTN_NLA;
  if (nla && (a->conv_w || a->qk_l2norm)) return GLINATTN_ERR_UNSUPPORTED;
  if (nla && (!a->z_pool || !aligned16(a->z_pool))) return GLINATTN_ERR_INVALID_ARG;
  if (!a->q || !a->k || !a->v || (!a->alpha && !nla) || !a->state_pool || !a->slot_ids || !a->accept)
    return GLINATTN_ERR_INVALID_ARG;
  if (a->variant == GLINATTN_GDN && !a->beta) return GLINATTN_ERR_INVALID_ARG;
  if (a->conv_w && !a->conv_pool) return GLINATTN_ERR_INVALID_ARG;
  if (!all_aligned(a->q, a->k, a->v, a->alpha, a->beta, a->state_pool, a->conv_w, a->conv_pool))
    return GLINATTN_ERR_INVALID_ARG;
  RecurParams p = {};
  p.variant = a->variant;
  p.in_bf16 = a->in_dtype == GLINATTN_BF16;
  p.qk_l2norm = a->qk_l2norm != 0;
  p.N = a->num_req;
  p.steps = a->draft_len;
  p.H = a->heads;
  p.Hq = Hq;
  p.pool_slots = a->pool_slots;
  p.Cch = a->heads * (2 * a->dk + a->dv);
  p.q = a->q;
  p.k = a->k;
  p.v = a->v;
  p.alpha = nla ? nullptr : a->alpha;
  p.beta = a->beta;
  p.S_src = a->state_pool;
  p.z_src = nla ? a->z_pool : nullptr;
  p.z_dst = nla ? a->z_pool : nullptr;
  p.src_slot = a->slot_ids;
  p.S_dst = a->state_pool;  // in place, the final state only
  p.dst_slot = a->slot_ids;
  p.dst_per_step = 0;
  p.step_count = a->accept;
  p.o = nullptr;
  p.conv_w = a->conv_w;
  p.conv_src = a->conv_w ? a->conv_pool : nullptr;
  p.conv_dst = a->conv_w ? a->conv_pool : nullptr;
  p.dev_status = a->dev_status;
  return glinattn::launch_recurrent(p, a->dk, a->dv, (cudaStream_t)stream);
}

}  // extern "C"
