// prefill_tc.cuh -- tensor-core (tcgen05 / TMEM / TMA) chunked prefill.
#pragma once

#include <cuda_runtime.h>

#include "glinattn.h"

namespace glinattn {

// True when the chunked tensor-core kernels are built into this library.
bool prefill_tc_available();

// Whether the tensor-core kernels cover this (validated) call.
bool prefill_tc_supports(const glinattn_prefill_args &a);

// bf16 activations, dk == dv == 128, chunk 64.  Arguments already validated.
glinattn_status launch_prefill_tc(const glinattn_prefill_args &a, cudaStream_t stream);

}  // namespace glinattn
