// static_scratch.cu -- a prefill entry point that allocates nothing.
//
// glinattn_prefill asks its caller for scratch space (the two-pass chunked
// Gated DeltaNet kernels keep per-chunk products there).  Some callers cannot
// provide it: a serving engine that plans all device memory up front -- the
// paged KV pool and the per-request state pool sized together against the
// request-length mix -- hands out no further device memory and does not let a
// library call cudaMalloc behind its back.  This entry point serves them from
// a fixed array in the library's own device image instead.
#include <cuda_runtime.h>

#include <mutex>

#include "glinattn.h"

namespace {

// The largest scratch the entry point can serve.  Chunked Gated DeltaNet
// prefill needs about 1.3 KB per (batch, head, token), so 32 MiB covers about
// 26,000 such positions per call (for example 16 heads x 1,600 tokens).
constexpr size_t kStaticScratchBytes = (size_t)32 << 20;

// Every GPU that loads the library holds this array until the process exits.
// In host code `g_static_scratch` names a host-side stand-in, not the device
// array: kernels only ever receive the address from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_lock;
void *g_scratch_addr[kMaxDevices];  // per device; nullptr until set up

// Device address of the array on the current device, looked up once per
// device with that device current.
glinattn_status scratch_address(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GLINATTN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return GLINATTN_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> guard(g_setup_lock);
  if (!g_scratch_addr[dev]) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || !ptr) return GLINATTN_ERR_CUDA;
    g_scratch_addr[dev] = ptr;
  }
  *out = g_scratch_addr[dev];
  return GLINATTN_OK;
}

}  // namespace

extern "C" glinattn_status glinattn_prefill_static_scratch(const glinattn_prefill_args *args,
                                                           glinattn_stream_t stream) {
  if (!args) return GLINATTN_ERR_INVALID_ARG;
  if (glinattn_prefill_workspace_size(args) > kStaticScratchBytes) return GLINATTN_ERR_UNSUPPORTED;
  void *scratch = nullptr;
  const glinattn_status st = scratch_address(&scratch);
  if (st != GLINATTN_OK) return st;
  glinattn_prefill_args a = *args;
  a.workspace = scratch;
  a.workspace_bytes = kStaticScratchBytes;
  return glinattn_prefill(&a, stream);
}
