/*
 * glinattn.h -- C ABI of the GB300 (sm_103a) state-passing linear-attention
 * layer: gated linear attention (GLA) and Gated DeltaNet (GDN).
 *
 * Source: "Inference for linear attention and hybrid architectures"
 * (ai-infra-handbooks):
 *   - section "Two ways to write the same computation": the two recurrences,
 *       GLA  S_t = alpha_t S_{t-1} + k_t^T v_t
 *       GDN  S_t = alpha_t (I - beta_t k_t^T k_t) S_{t-1} + beta_t k_t^T v_t
 *     with o_t = q_t S_t read after the update; the chunked form used for
 *     prefill; the hand-over of the state between prefill segments; the short
 *     causal convolution in front of the layer and its per-request cache;
 *   - section "A new memory ledger": a per-request state pool, states in fp32;
 *   - section "Speculative decoding and PD disaggregation": one state per
 *     draft position for rollback; batched kernels read and write the state
 *     pool by slot index.
 *
 * Conventions shared by every call
 *   - All tensor arguments are DEVICE pointers to caller-owned memory,
 *     contiguous row-major in the layout stated (innermost index last), with
 *     the base address 16-byte aligned.  The library keeps no pointer after
 *     the call returns and allocates no device memory; scratch space, where a
 *     kernel needs it, is passed in by the caller (glinattn_prefill_workspace_size).
 *   - Calls are asynchronous on the given stream (0 = legacy default stream).
 *     Argument errors are detected on the host before anything is launched and
 *     returned as a status; the output buffers are then untouched.
 *   - dev_status (nullable) is a device word the kernels OR error bits into
 *     (GLINATTN_DEV_*); a unit that raises a bit skips its writes.  The caller
 *     zeroes it and reads it after synchronising.
 *   - Head sizes: dk == dv, one of 16, 32, 64, 128; or dk = 128, dv = 64, the
 *     SSD form of Mamba2 (state size 128, head dim 64: "Long context, fast
 *     inference, smart decoding, and life beyond attention", section
 *     "Mamba and hybrid SSMs, the real packages"; the linear-attention page's
 *     section "Two ways to write the same computation" lists the SSD form
 *     among the gated linear attention recurrences).  Activations (q, k, v,
 *     conv cache) are all GLINATTN_BF16 or all GLINATTN_F32; gates alpha and
 *     beta, states and conv weights are fp32.  alpha must lie in (0, 1],
 *     beta in [0, 1].
 *   - The short convolution is depthwise, width 4, over the channels
 *     [q | k | v] of every head, Cch = H * (2 dk + dv) channels, channel index
 *     part_offset + h * d + i.  Weight w[c][j] multiplies input x_{t-3+j}
 *     (tap 3 is the current token); no bias, no activation.  The conv cache
 *     holds the last 3 RAW inputs per channel, oldest first: [.., 3, Cch].
 *   - Grouped q / k heads (qk_heads = Hq, 0 meaning Hq = H): q and k are
 *     [.., Hq, dk] and consecutive groups of H / Hq heads share them, head h
 *     reading q / k head h / (H / Hq) (the SSD form's B and C shared by the
 *     heads of a group).  Hq must divide H; grouped heads take no
 *     convolution (GLINATTN_ERR_UNSUPPORTED).  Everything else stays per head.
 *   - qk_l2norm != 0 rescales each q and k row of each head to
 *     x / sqrt(sum x^2 + 1e-6) after the convolution.  With bf16 activations
 *     the convolved / normalised values are rounded to bf16 before use.
 */
#ifndef GLINATTN_H
#define GLINATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *glinattn_stream_t; /* a cudaStream_t */

typedef enum {
  GLINATTN_OK = 0,
  GLINATTN_ERR_INVALID_ARG = 1, /* null pointer, bad size, misalignment, aliasing */
  GLINATTN_ERR_UNSUPPORTED = 2, /* valid but not built: head size, dtype combination */
  GLINATTN_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed (launch, attribute) */
  GLINATTN_ERR_DEVICE_STATUS = 4, /* reserved for host helpers that read dev_status */
  GLINATTN_ERR_TIMEOUT = 5      /* reserved: a bounded device wait gave up */
} glinattn_status;

/*
 * GLINATTN_NLA: normalised kernelised linear attention ("Long context, fast
 * inference, smart decoding, and life beyond attention", section "Linear
 * attention: removing softmax entirely"): with phi(x) = elu(x) + 1 applied to
 * q and k inside the layer,
 *   S_t = S_{t-1} + phi(k_t)^T v_t,  z_t = z_{t-1} + phi(k_t),
 *   o_t = phi(q_t) S_t / (phi(q_t) . z_t + 1e-6).
 * No gates (alpha and beta are ignored and may be NULL), no convolution, no
 * L2 norm; the normaliser z [.., H, dk] fp32 travels beside the state.
 */
typedef enum { GLINATTN_GLA = 0, GLINATTN_GDN = 1, GLINATTN_NLA = 2 } glinattn_variant;
typedef enum { GLINATTN_F32 = 0, GLINATTN_BF16 = 1 } glinattn_dtype;

/* Bits OR-ed into *dev_status by the kernels. */
#define GLINATTN_DEV_BAD_SLOT 0x1u    /* slot id outside [0, pool_slots): unit skipped */
#define GLINATTN_DEV_BAD_GATE 0x2u    /* alpha outside (0, 1] or not finite: unit skipped */
#define GLINATTN_DEV_WAIT_TIMEOUT 0x4u /* an on-chip barrier wait exceeded its bound */
#define GLINATTN_DEV_BAD_COUNT 0x8u   /* accepted length outside [0, draft_len]: request skipped */

/*
 * glinattn_prefill -- chunked prefill of one segment for B sequences.
 *   Computes o_t = q_t S_t for t = 1..T and the final state S_T of every
 *   (sequence, head), starting from S0 (or zeros) and the conv cache conv_in
 *   (or zero history).  Feeding S_T and conv_out of one call as S0 and
 *   conv_in of the next continues the sequence exactly (segmented prefill).
 *
 *   q, k   [B, T, Hq, dk]  v [B, T, H, dv]       activations (in_dtype)
 *   alpha  [B, T, H]       beta [B, T, H] (GDN only, else NULL)       fp32
 *   S0     [B, H, dk, dv]  fp32 or NULL (zero state)
 *   S_T    [B, H, dk, dv]  fp32 output; may alias S0 exactly
 *   o      [B, T, H, dv]   output (out_dtype)
 *   conv_w [Cch, 4] fp32 or NULL (no convolution; conv_in/conv_out ignored)
 *   conv_in  [B, 3, Cch] (in_dtype) or NULL (zero history)
 *   conv_out [B, 3, Cch] (in_dtype) or NULL; may alias conv_in exactly
 *   T may be any value >= 0 (a ragged last chunk is handled); T == 0 copies
 *   S0 to S_T and conv_in to conv_out.
 *   state_every > 0 also emits the state at block boundaries for prefix
 *   caching (section "Prefix caching has to be redone": a prefix can be
 *   reused only where its state was kept): S_blocks [B, T / state_every, H,
 *   dk, dv] fp32 receives the state after token j * state_every of this
 *   segment, j = 1 .. T / state_every (rounded down).  The chunked kernels
 *   need state_every to be a multiple of the chunk (64), else the call returns
 *   GLINATTN_ERR_UNSUPPORTED; the fp32 token-serial kernel takes any value.
 *   0 emits nothing and S_blocks is ignored.  With a convolution, conv_blocks
 *   (when not NULL) [B, T / state_every, 3, Cch] (in_dtype) receives the conv
 *   cache at the same boundaries, so that (S_blocks[:, j], conv_blocks[:, j])
 *   is a whole checkpoint a later prefill or decode can start from.
 *   bf16 activations with dk = 128 run the tensor-core chunked kernels (chunk
 *   64): gated linear attention with dv = 128 or 64, grouped q / k heads
 *   allowed, no convolution or L2 norm; Gated DeltaNet with dv = 128 and one
 *   q / k head per head (it also needs `workspace`, see below, else
 *   GLINATTN_ERR_INVALID_ARG).  Every other supported combination runs the
 *   fp32 token-serial kernel, which is exact to fp32 rounding but not fast.
 */
typedef struct {
  int32_t variant;   /* glinattn_variant */
  int32_t in_dtype;  /* glinattn_dtype of q, k, v, conv cache */
  int32_t out_dtype; /* glinattn_dtype of o */
  int32_t qk_l2norm;
  int32_t batch, seqlen, heads, dk, dv;
  int32_t state_every; /* 0, or the block length of emitted states (see above) */
  const void *q, *k, *v;
  const float *alpha, *beta;
  const float *S0;
  float *S_T;
  void *o;
  const float *conv_w;
  const void *conv_in;
  void *conv_out;
  uint32_t *dev_status;
  void *workspace;        /* device scratch, >= glinattn_prefill_workspace_size() bytes */
  size_t workspace_bytes; /* its size; may be 0 when the size query returns 0 */
  float *S_blocks;        /* [B, T / state_every, H, dk, dv] fp32 when state_every > 0 */
  void *conv_blocks;      /* [B, T / state_every, 3, Cch] (in_dtype) or NULL */
  int32_t qk_heads;       /* q / k heads Hq (0: Hq = H), see "Grouped q / k heads" above */
  const float *z0;        /* GLINATTN_NLA: normaliser in [B, H, dk] fp32, or NULL (zeros) */
  float *z_T;             /* GLINATTN_NLA: normaliser out [B, H, dk] fp32 (may alias z0) */
} glinattn_prefill_args;

glinattn_status glinattn_prefill(const glinattn_prefill_args *args, glinattn_stream_t stream);

/*
 * glinattn_prefill_workspace_size -- bytes of device scratch the call needs
 *   for these arguments (only sizes, variant and dtypes are read).  The
 *   caller owns the buffer; calls on one stream may reuse it.  Nonzero for:
 *   - chunked Gated DeltaNet (required): a parallel pass over all chunks
 *     stores the front-end outputs q', k', the state-independent chunk
 *     products W = (I+A)^-1 diag(beta gamma) K' and U~ = (I+A)^-1 diag(beta) V'
 *     and the gates there, about 1.3 KB per (batch, head, token); the serial
 *     pass reads them;
 *   - chunked normalised linear attention (required): the features, the
 *     chunk sums of phi(k) and a copy of the start normaliser;
 *   - chunked gated linear attention when so few (batch, head) units would
 *     leave more than half of the SMs idle (optional): with the scratch the
 *     sequence is split into pieces -- a pass computes every piece's end
 *     state from a zero start, a combine gives every piece its start state,
 *     and the usual kernel then runs the pieces in parallel.  Without it (or
 *     with a smaller one) the call runs the unsplit kernel; both orders of
 *     summation are within the stated tolerance but can differ in the last
 *     bits.
 *   Every other configuration needs 0 bytes.
 */
size_t glinattn_prefill_workspace_size(const glinattn_prefill_args *args);

/*
 * glinattn_prefill_static_scratch -- glinattn_prefill for callers that cannot
 *   allocate device memory.  The source pages have no counterpart: this is a
 *   deployment interface, not part of the method.  A serving engine that plans
 *   all of its device memory up front (the paged KV pool and the per-request
 *   state pool, sized together against the request-length mix) has no spare
 *   buffer to pass as `workspace` and does not let a library call cudaMalloc;
 *   this entry point takes its scratch from a fixed 32 MiB array in the
 *   library's device image instead.
 *
 *   - args->workspace and args->workspace_bytes are ignored; every other field
 *     means what it means for glinattn_prefill, with the same validation.  The
 *     results are bit for bit those of glinattn_prefill given a workspace of
 *     at least glinattn_prefill_workspace_size() bytes (for gated linear
 *     attention with few units that is the split path, see above).
 *   - A call whose glinattn_prefill_workspace_size() exceeds 32 MiB (about
 *     26,000 batch x head x token positions of chunked Gated DeltaNet prefill)
 *     returns GLINATTN_ERR_UNSUPPORTED and launches nothing.
 *   - It calls no cudaMalloc or cudaFree.  The array exists once per GPU that
 *     loads the library and stays allocated until the process exits.  The
 *     first call on a device looks up the array's device address on that
 *     device (cudaGetSymbolAddress, with the device current); make that first
 *     call before any stream capture.
 *   - Every call shares the one array, which keeps the previous call's
 *     contents (the kernels overwrite every byte they read, so nothing needs
 *     clearing).  Calls that may overlap on the GPU -- on different streams,
 *     or from different host threads -- race on it: serialise them.
 */
glinattn_status glinattn_prefill_static_scratch(const glinattn_prefill_args *args,
                                                glinattn_stream_t stream);

/*
 * glinattn_decode -- one recurrent decode step for N requests.
 *   For request n with slot s = slot_ids[n]: runs the conv step against
 *   conv_pool[s] (then shifts it), reads state_pool[s], applies one rank-one
 *   update, writes the state back IN PLACE and writes o[n].  Slots not named
 *   in slot_ids are not touched.  slot_ids must be distinct (not checked on
 *   the device: duplicates race); ids outside [0, pool_slots) set
 *   GLINATTN_DEV_BAD_SLOT and skip that request.
 *
 *   q, k [N, Hq, dk]   v [N, H, dv]   alpha, beta [N, H]   slot_ids [N] int32
 *   state_pool [P, H, dk, dv] fp32 (read/write)   o [N, H, dv]
 *   conv_w [Cch, 4] or NULL;  conv_pool [P, 3, Cch] (in_dtype, read/write)
 */
typedef struct {
  int32_t variant, in_dtype, out_dtype, qk_l2norm;
  int32_t num_req, heads, dk, dv, pool_slots;
  int32_t qk_heads; /* q / k heads Hq (0: Hq = H) */
  const void *q, *k, *v;
  const float *alpha, *beta;
  float *state_pool;
  const int32_t *slot_ids;
  void *o;
  const float *conv_w;
  void *conv_pool;
  uint32_t *dev_status;
  float *z_pool; /* GLINATTN_NLA: normalisers [P, H, dk] fp32, indexed like state_pool */
} glinattn_decode_args;

glinattn_status glinattn_decode(const glinattn_decode_args *args, glinattn_stream_t stream);

/*
 * glinattn_spec_decode -- speculative decode of D draft tokens per request,
 *   keeping one state per draft position.  Starting from state_pool[src_slots[n]]
 *   (and its conv cache), step i = 0..D-1 consumes draft token i and writes the
 *   state after it to state_pool[dst_slots[n*D + i]] (and the conv cache to the
 *   same slot of conv_pool); o[n, i] is its output.  The source slot is only
 *   read.  Rolling back to an accepted prefix of length a is the caller's
 *   choice of slot: src_slots[n] for a = 0, else dst_slots[n*D + a - 1]; the
 *   state there is bit-identical to a decode steps of glinattn_decode.
 *   All destination slots of all requests must be distinct from each other
 *   and from every source slot (not checked on the device).
 *   dst_slots == NULL verifies only: the outputs are written, no state and no
 *   conv cache, and the pool keeps one state per request; glinattn_replay
 *   then applies the accepted drafts (the replay-buffer alternative).  For
 *   GLA and Gated DeltaNet with dk = dv = 128, q / k heads = heads and
 *   draft_len <= 16, the verify-only outputs come from the chunked form of
 *   the section "Two ways to write the same computation" over the D drafts
 *   (one read of the start state), so they equal the per-draft outputs up to
 *   fp32 rounding rather than bit for bit; the front end (conv, L2 norm, bf16
 *   rounding of q, k, v) is the decode step's, bit for bit.
 *
 *   q, k [N, D, Hq, dk]   v [N, D, H, dv]   alpha, beta [N, D, H]
 *   src_slots [N]  dst_slots [N, D] or NULL  int32    o [N, D, H, dv]
 */
typedef struct {
  int32_t variant, in_dtype, out_dtype, qk_l2norm;
  int32_t num_req, draft_len, heads, dk, dv, pool_slots;
  const void *q, *k, *v;
  const float *alpha, *beta;
  float *state_pool;
  const int32_t *src_slots;
  const int32_t *dst_slots;
  void *o;
  const float *conv_w;
  void *conv_pool;
  uint32_t *dev_status;
  int32_t qk_heads; /* q / k heads Hq (0: Hq = H) */
  float *z_pool; /* GLINATTN_NLA: normalisers [P, H, dk] fp32, indexed like state_pool */
} glinattn_spec_args;

glinattn_status glinattn_spec_decode(const glinattn_spec_args *args, glinattn_stream_t stream);

/*
 * glinattn_replay -- roll the pool forward over the accepted drafts, the
 *   alternative to keeping one state per draft position (section "Speculative
 *   decoding and PD disaggregation": the updates of the draft steps are
 *   recorded and replayed from a chosen position).  The recorded draft inputs
 *   of a verify-only glinattn_spec_decode are the replay buffer: for request
 *   n, the first accept[n] draft steps are applied to state_pool[slot_ids[n]]
 *   and its conv cache, in place, with the arithmetic of glinattn_decode, so
 *   the result equals accept[n] decode steps (and the per-draft state of
 *   glinattn_spec_decode) bit for bit.  accept[n] == 0 leaves the slot as it
 *   is; a length outside [0, D] sets GLINATTN_DEV_BAD_COUNT and skips the
 *   request; slot ids outside [0, pool_slots) set GLINATTN_DEV_BAD_SLOT.
 *   Only the applied steps' gates are checked.  No outputs are written.
 *
 *   q, k [N, D, Hq, dk]   v [N, D, H, dv]   alpha, beta [N, D, H]   (in_dtype / fp32)
 *   slot_ids [N] int32 (distinct)   accept [N] int32
 *   state_pool [P, H, dk, dv] fp32 and conv_pool [P, 3, Cch] (read/write)
 */
typedef struct {
  int32_t variant, in_dtype, qk_l2norm;
  int32_t num_req, draft_len, heads, dk, dv, pool_slots;
  int32_t qk_heads; /* q / k heads Hq (0: Hq = H) */
  const void *q, *k, *v;
  const float *alpha, *beta;
  float *state_pool;
  const int32_t *slot_ids;
  const int32_t *accept;
  const float *conv_w;
  void *conv_pool;
  uint32_t *dev_status;
  float *z_pool; /* GLINATTN_NLA: normalisers [P, H, dk] fp32, indexed like state_pool */
} glinattn_replay_args;

glinattn_status glinattn_replay(const glinattn_replay_args *args, glinattn_stream_t stream);

/*
 * glinattn_state_copy -- copy whole slots of a state pool (and of its conv
 *   cache pool): for i < n, state_pool[dst_slots[i]] = state_pool[src_slots[i]]
 *   and, when conv_pool is given, conv_pool[dst_slots[i]] =
 *   conv_pool[src_slots[i]].  Section "Prefix caching has to be redone": a
 *   request that reuses a cached prefix starts from a copy of the prefix's
 *   state, never from the cached slot itself (copy on write); section
 *   "Speculative decoding and PD disaggregation": an accepted draft's state
 *   can be copied back to the request's own slot.
 *
 *   state_pool [P, H, dk, dv] fp32     conv_pool [P, 3, Cch] (in_dtype) or NULL
 *   src_slots, dst_slots [n] int32 (device memory)
 *   A pair whose slot is outside [0, pool_slots) is skipped and raises
 *   GLINATTN_DEV_BAD_SLOT in *dev_status (when given).  Destination slots must
 *   be distinct and must not be a source slot of another pair of the same call
 *   (not checked on the device).
 */
typedef struct {
  int32_t n, pool_slots, heads, dk, dv, in_dtype;
  float *state_pool;
  void *conv_pool;
  const int32_t *src_slots;
  const int32_t *dst_slots;
  uint32_t *dev_status;
} glinattn_copy_args;

glinattn_status glinattn_state_copy(const glinattn_copy_args *args, glinattn_stream_t stream);

/*
 * glinattn_selective_scan -- Mamba's selective state-space scan over one
 *   segment ("Long context, fast inference, smart decoding, and life beyond
 *   attention", chapter "05 · State-space models: the architectural
 *   alternative", section "Mamba: making the recurrence input-dependent, and
 *   the engineering that makes that fast anyway").  For channel d and state
 *   index n, with dt = softplus(delta) = log(1 + e^delta):
 *     h_t[d, n] = exp(dt_t[d] A[d, n]) h_{t-1}[d, n] + dt_t[d] Bm_t[n] x_t[d]
 *     y_t[d]    = sum_n h_t[d, n] Cm_t[n]
 *   The projections producing delta, Bm and Cm are the caller's; the scan
 *   applies the softplus.  All arithmetic is fp32.
 *
 *   x, delta [B, T, D] and Bm, Cm [B, T, N]   (in_dtype)
 *   A [D, N] fp32     h0 [B, D, N] fp32 or NULL (zeros)
 *   h_T [B, D, N] fp32 output (may alias h0 exactly)     y [B, T, D] (out_dtype)
 *   N (state) in {8, 16, 32}; any D >= 1.  T == 0 copies h0 to h_T.
 *   workspace: at least glinattn_selective_scan_workspace_size() bytes (the
 *   chunk end states, step sums and start states), 16-byte aligned.
 */
typedef struct {
  int32_t in_dtype, out_dtype;
  int32_t batch, seqlen, channels, state;
  const void *x, *delta, *Bm, *Cm;
  const float *A;
  const float *h0;
  float *h_T;
  void *y;
  void *workspace;
  size_t workspace_bytes;
  uint32_t *dev_status;
} glinattn_scan_args;

size_t glinattn_selective_scan_workspace_size(const glinattn_scan_args *args);
glinattn_status glinattn_selective_scan(const glinattn_scan_args *args, glinattn_stream_t stream);

/*
 * glinattn_selective_scan_decode -- one step of the selective scan for R
 *   requests, the states in a slot-indexed pool updated in place:
 *   state_pool[slot_ids[r]] is h of request r.  An id outside
 *   [0, pool_slots) sets GLINATTN_DEV_BAD_SLOT and skips the request; ids must
 *   be distinct.
 *
 *   x, delta [R, D]   Bm, Cm [R, N]   (in_dtype)    A [D, N] fp32
 *   state_pool [P, D, N] fp32 (read/write)   slot_ids [R] int32   y [R, D] (out_dtype)
 */
typedef struct {
  int32_t in_dtype, out_dtype;
  int32_t num_req, channels, state, pool_slots;
  const void *x, *delta, *Bm, *Cm;
  const float *A;
  float *state_pool;
  const int32_t *slot_ids;
  void *y;
  uint32_t *dev_status;
} glinattn_scan_decode_args;

glinattn_status glinattn_selective_scan_decode(const glinattn_scan_decode_args *args, glinattn_stream_t stream);

/* Human-readable name of a status code (static storage). */
const char *glinattn_status_string(glinattn_status status);

/* Library version, major * 10000 + minor * 100 + patch. */
int glinattn_version(void);

/* Bytes of one request's state in one layer: heads * dk * dv * 4. */
size_t glinattn_state_bytes(int heads, int dk, int dv);

#ifdef __cplusplus
}
#endif

#endif /* GLINATTN_H */
