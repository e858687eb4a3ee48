// common.cuh -- small internals shared by the glinattn CUDA translation units.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "glinattn.h"

namespace glinattn {

// Kernel parameters of the token-serial recurrent kernel (decode, speculative
// decode and the fp32 prefill path).  A "unit" is one (request, head) pair;
// every unit consumes `steps` tokens laid out [N, steps, H, d].
struct RecurParams {
  int variant, in_bf16, out_bf16, qk_l2norm;
  int N, steps, H, pool_slots;  // pool_slots = 0 when states are not pooled
  int Hq;                       // q / k heads (groups of H / Hq heads share them)
  int Cch;                      // conv channels per request, H * 3d
  const void *q, *k, *v;
  const float *alpha, *beta;
  // state source: S_src + (slot or n) * H*d*d + h*d*d; NULL means zeros
  const float *S_src;
  // normalised linear attention: normaliser source / destination, indexed
  // like the states ([.., H, dk] fp32)
  const float *z_src;
  float *z_dst;
  const int32_t *src_slot;  // [N] or NULL (index by n)
  // state destination(s)
  float *S_dst;
  const int32_t *dst_slot;  // [N] (final) or [N*steps] (per step) or NULL (index by n)
  int dst_per_step;
  void *o;
  // short convolution: weights [Cch, 4]; caches [.., 3, Cch] indexed like the states
  const float *conv_w;
  const void *conv_src;  // NULL = zero history
  void *conv_dst;        // NULL = not written
  uint32_t *dev_status;
  // [N] steps applied per request (0 .. steps; NULL: all): the replay of
  // accepted drafts.  With S_dst == NULL no state or conv cache is written,
  // with o == NULL no output.
  const int32_t *step_count;
  // prefill only: the state after every state_every tokens to S_blocks
  // [N, nblocks, H, d, d] (state_every == 0: none)
  float *S_blocks;
  int state_every, nblocks;
};

glinattn_status launch_recurrent(const RecurParams &p, int dk, int dv, cudaStream_t stream);
// conv caches at the emitted block boundaries of a prefill (checkpoint.cu)
glinattn_status launch_conv_blocks(const glinattn_prefill_args &a, cudaStream_t stream);

// Persistent pipelined decode / speculative decode for 128 x 128 pooled states.
bool decode128_supports(const RecurParams &p, int d);
cudaError_t launch_decode128(const RecurParams &p, cudaStream_t stream);
// Verify-only speculative decode (outputs, no states) from one read of each
// start state, in the chunked form over the drafts.
bool verify128_supports(const RecurParams &p, int d);
cudaError_t launch_verify128(const RecurParams &p, cudaStream_t stream);

}  // namespace glinattn
