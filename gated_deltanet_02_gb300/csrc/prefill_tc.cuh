// prefill_tc.cuh -- tensor-core (tcgen05 / TMEM / TMA) chunked prefill.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>

#include "glinattn.h"

namespace glinattn {

// True when the chunked tensor-core kernels are built into this library.
bool prefill_tc_available();

// Whether the tensor-core kernels cover this (validated) call.
bool prefill_tc_supports(const glinattn_prefill_args &a);

// bf16 activations, dk == dv == 128, chunk 64.  Arguments already validated.
glinattn_status launch_prefill_tc(const glinattn_prefill_args &a, cudaStream_t stream);
// The same with a per-unit skip flag array [B, H] (NULL: none).
glinattn_status launch_prefill_tc_skip(const glinattn_prefill_args &a, cudaStream_t stream, const int *skip);
// The same kernel for normalised linear attention (nonzero dz): q and k are
// the features, no gates; dz [B, Hq, nchunks, d_k] holds every chunk's column
// sums of phi(k), z0 [B, H, d_k] the start normaliser (not overlapping z_T),
// z_T [B, H, d_k] receives the final one (NULL: not written), and the outputs
// are divided by phi(q_t) . z_t + 1e-6.
glinattn_status launch_prefill_tc_nla(const glinattn_prefill_args &a, cudaStream_t stream, const int *skip,
                                      const float *dz, const float *z0, float *z_T);

// Gated linear attention split along the sequence when B * H * (d_v / 64)
// leaves more than half of the SMs idle (gla_split.cu): the number of pieces
// (1 = no split), the workspace it needs, and the launch.
int gla_split_pieces(const glinattn_prefill_args &a);
size_t gla_split_workspace_bytes(const glinattn_prefill_args &a);
glinattn_status launch_gla_split(const glinattn_prefill_args &a, cudaStream_t stream);

// Chunked Gated DeltaNet (two passes through a caller-provided workspace).
bool gdn_tc_supports(const glinattn_prefill_args &a);
size_t gdn_tc_workspace_bytes(const glinattn_prefill_args &a);
glinattn_status launch_gdn_tc(const glinattn_prefill_args &a, cudaStream_t stream);

// Chunked normalised linear attention (features, z at chunk starts, then the
// gate-free chunked kernel dividing in its epilogue) through a caller-provided
// workspace.
bool nla_tc_supports(const glinattn_prefill_args &a);
size_t nla_tc_workspace_bytes(const glinattn_prefill_args &a);
glinattn_status launch_nla_tc(const glinattn_prefill_args &a, cudaStream_t stream);

// [B, T, H, d] bf16 activations as a 4-D map (d, H, T, B); box 64 x 1 x 64 x 1
// (64 channels of one head for 64 tokens), 128-byte swizzle.
bool make_act_map(CUtensorMap *m, const void *base, int B, int T, int H, int d);

// General 3-D tiled map: dims (innermost first) and box in elements.
bool encode_3d_map(CUtensorMap *m, const void *base, CUtensorMapDataType type, int elem_bytes,
                   const long long dims[3], const int box[3], bool swizzle);

// 3-D tiled map over rows of `inner` elements: dims (inner, rows, planes),
// box (box_inner, 64, 1); 128-byte swizzle when `swizzle` is set.
bool encode_rows_map(CUtensorMap *m, const void *base, CUtensorMapDataType type, int elem_bytes,
                     int inner, int rows, int planes, int box_inner, bool swizzle);

}  // namespace glinattn
