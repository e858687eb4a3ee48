// prefill_tc.cu -- placeholder until the tensor-core kernels land.
#include "prefill_tc.cuh"

namespace glinattn {
bool prefill_tc_available() { return false; }
glinattn_status launch_prefill_tc(const glinattn_prefill_args &, cudaStream_t) {
  return GLINATTN_ERR_UNSUPPORTED;
}
}  // namespace glinattn
