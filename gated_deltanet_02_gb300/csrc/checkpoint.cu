// checkpoint.cu -- prefix-cache checkpoints: whole-slot copies inside a state
// pool (and its conv pool), and the conv history at emitted block boundaries.
//
// "Inference for linear attention and hybrid architectures", section "Prefix
// caching has to be redone": a state summarises its whole prefix, so a prefix
// can be reused only where a checkpoint (state plus conv cache) was kept, and a
// request that reuses it starts from its own copy (copy on write), because
// decoding overwrites the state in place.  Section "Speculative decoding and PD
// disaggregation": the state of an accepted draft can be copied back into the
// request's own slot.  A slot is H * dk * dv fp32 values (1 MiB for 16 heads of
// 128 x 128), so the copy is a plain streaming kernel: one grid row per pair,
// 16-byte loads and stores, coalesced.
#include "common.cuh"

namespace glinattn {
namespace {

constexpr int kCopyThreads = 256;

__global__ void __launch_bounds__(kCopyThreads)
    slot_copy_kernel(float *pool, size_t slot_floats, void *conv_pool, size_t conv_bytes, int pool_slots,
                     const int32_t *src_slots, const int32_t *dst_slots, uint32_t *dev_status) {
  const int i = blockIdx.y;
  const int src = src_slots[i], dst = dst_slots[i];
  if (src < 0 || src >= pool_slots || dst < 0 || dst >= pool_slots) {
    if (blockIdx.x == 0 && threadIdx.x == 0 && dev_status) atomicOr(dev_status, GLINATTN_DEV_BAD_SLOT);
    return;
  }
  const size_t n4 = slot_floats / 4;  // slot_floats is a multiple of 4
  const float4 *s4 = reinterpret_cast<const float4 *>(pool + (size_t)src * slot_floats);
  float4 *d4 = reinterpret_cast<float4 *>(pool + (size_t)dst * slot_floats);
  const size_t stride = (size_t)gridDim.x * kCopyThreads;
  for (size_t j = (size_t)blockIdx.x * kCopyThreads + threadIdx.x; j < n4; j += stride) d4[j] = s4[j];
  if (conv_pool) {  // conv_bytes is a multiple of 16
    const uint4 *c_s = reinterpret_cast<const uint4 *>(static_cast<const uint8_t *>(conv_pool) + (size_t)src * conv_bytes);
    uint4 *c_d = reinterpret_cast<uint4 *>(static_cast<uint8_t *>(conv_pool) + (size_t)dst * conv_bytes);
    for (size_t j = (size_t)blockIdx.x * kCopyThreads + threadIdx.x; j < conv_bytes / 16; j += stride)
      c_d[j] = c_s[j];
  }
}

// The conv cache at the end of block j (tokens [0, (j + 1) * every)): the last
// three raw [q | k | v] rows before that point, oldest first, taken from the
// segment's inputs or, for positions before the segment, from conv_in (zeros
// when it is null).  Grid (nblocks, B); every row part is a whole number of
// 16-byte words.
__global__ void __launch_bounds__(kCopyThreads)
    conv_block_kernel(const uint8_t *q, const uint8_t *k, const uint8_t *v, const uint8_t *conv_in,
                      uint8_t *conv_blocks, int T, int every, int nblocks, size_t qk_bytes, size_t v_bytes) {
  const int j = blockIdx.x, b = blockIdx.y;
  const size_t row_bytes = 2 * qk_bytes + v_bytes;
  const int end = (j + 1) * every;
  for (int r = 0; r < 3; ++r) {
    const int pos = end - 3 + r;
    uint4 *dst = reinterpret_cast<uint4 *>(conv_blocks + (((size_t)b * nblocks + j) * 3 + r) * row_bytes);
    const size_t nw = row_bytes / 16, nqk = qk_bytes / 16;
    for (size_t w = threadIdx.x; w < nw; w += kCopyThreads) {
      uint4 x = make_uint4(0, 0, 0, 0);
      if (pos >= 0) {
        const size_t tok = (size_t)b * T + pos;
        if (w < nqk) x = reinterpret_cast<const uint4 *>(q + tok * qk_bytes)[w];
        else if (w < 2 * nqk) x = reinterpret_cast<const uint4 *>(k + tok * qk_bytes)[w - nqk];
        else x = reinterpret_cast<const uint4 *>(v + tok * v_bytes)[w - 2 * nqk];
      } else if (conv_in) {
        x = reinterpret_cast<const uint4 *>(conv_in + ((size_t)b * 3 + 3 + pos) * row_bytes)[w];
      }
      dst[w] = x;
    }
  }
}

}  // namespace

glinattn_status launch_conv_blocks(const glinattn_prefill_args &a, cudaStream_t stream) {
  const int every = a.state_every, nblocks = a.seqlen / every;
  const size_t esz = a.in_dtype == GLINATTN_BF16 ? 2 : 4;
  const size_t qk_bytes = (size_t)a.heads * a.dk * esz, v_bytes = (size_t)a.heads * a.dv * esz;
  if (qk_bytes % 16 || v_bytes % 16) return GLINATTN_ERR_UNSUPPORTED;
  if (a.batch > 65535) return GLINATTN_ERR_UNSUPPORTED;  // one grid row per sequence
  const dim3 grid((unsigned)nblocks, (unsigned)a.batch);
  conv_block_kernel<<<grid, kCopyThreads, 0, stream>>>(
      static_cast<const uint8_t *>(a.q), static_cast<const uint8_t *>(a.k), static_cast<const uint8_t *>(a.v),
      static_cast<const uint8_t *>(a.conv_in), static_cast<uint8_t *>(a.conv_blocks), a.seqlen, every, nblocks,
      qk_bytes, v_bytes);
  return cudaGetLastError() == cudaSuccess ? GLINATTN_OK : GLINATTN_ERR_CUDA;
}

}  // namespace glinattn

extern "C" glinattn_status glinattn_state_copy(const glinattn_copy_args *a, glinattn_stream_t stream) {
  if (!a) return GLINATTN_ERR_INVALID_ARG;
  if (a->n < 0 || a->pool_slots <= 0 || a->heads <= 0 || a->dk <= 0 || a->dv <= 0) return GLINATTN_ERR_INVALID_ARG;
  if (a->in_dtype != GLINATTN_F32 && a->in_dtype != GLINATTN_BF16) return GLINATTN_ERR_INVALID_ARG;
  if (a->n == 0) return GLINATTN_OK;
  if (a->n > 65535) return GLINATTN_ERR_UNSUPPORTED;  // one grid row per pair
  if (!a->state_pool || !a->src_slots || !a->dst_slots) return GLINATTN_ERR_INVALID_ARG;
  const size_t slot_floats = (size_t)a->heads * a->dk * a->dv;
  const size_t conv_bytes = (size_t)3 * a->heads * (2 * a->dk + a->dv) * (a->in_dtype == GLINATTN_BF16 ? 2 : 4);
  if (slot_floats % 4 != 0 || (a->conv_pool && conv_bytes % 16 != 0)) return GLINATTN_ERR_UNSUPPORTED;
  if (((uintptr_t)a->state_pool & 15u) || ((uintptr_t)a->conv_pool & 15u)) return GLINATTN_ERR_INVALID_ARG;
  // enough CTAs per pair to stream one slot at full width, at most 64
  size_t per = (slot_floats / 4 + glinattn::kCopyThreads * 4 - 1) / (glinattn::kCopyThreads * 4);
  if (per < 1) per = 1;
  if (per > 64) per = 64;
  const dim3 grid((unsigned)per, (unsigned)a->n);
  glinattn::slot_copy_kernel<<<grid, glinattn::kCopyThreads, 0, (cudaStream_t)stream>>>(
      a->state_pool, slot_floats, a->conv_pool, a->conv_pool ? conv_bytes : 0, a->pool_slots, a->src_slots,
      a->dst_slots, a->dev_status);
  return cudaGetLastError() == cudaSuccess ? GLINATTN_OK : GLINATTN_ERR_CUDA;
}
