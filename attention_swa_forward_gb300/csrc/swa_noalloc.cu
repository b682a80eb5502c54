// swa_noalloc.cu — swa_backward_noalloc: the backward for callers that cannot
// give the library device memory.
//
// Some callers cannot call cudaMalloc at the point where they run the
// backward: for example a plugin inside a host framework that owns all device
// memory through its own pool and forbids foreign allocations, or a
// latency-critical loop that must not allocate after start-up (cudaMalloc may
// synchronise the device and take milliseconds).  For them this entry point
// uses a fixed scratch area compiled into the library instead of a
// caller-supplied workspace.  The caller still passes every input and output.
//
// The scratch is one file-scope device array of kNoAllocScratchBytes.  Every
// GPU that loads this library holds it until the process exits, and every
// call on that GPU shares it: two calls whose kernels overlap on the GPU race
// on it.  Whatever must start at zero (the status word) is cleared on every
// call: by the backward's own first kernel, or by a memset in the
// bounds-checked build.
#include "swa.h"

#include <cuda_runtime.h>

#include "swa_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;  // 64 MiB

// Device-resident scratch.  In host code this name only stands in for the
// symbol; its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch in the current context, looked up on every
// call.  A cached address could outlive its context (after cudaDeviceReset,
// or under another context on the same device) and send the kernels to
// memory that is no longer the scratch; the lookup is cheap once the module
// is loaded.  The first lookup on a device may load the module, which is why
// the first call should come before any stream capture.
swa_status_t scratch_in_current_context(void** out) {
  void* ptr = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
  if (e != cudaSuccess || !ptr) {
    int dev = -1;
    cudaGetDevice(&dev);
    return swa::set_error(SWA_ERR_CUDA, "cudaGetSymbolAddress of the no-alloc scratch failed on device %d: %s", dev,
                          cudaGetErrorString(e));
  }
  *out = ptr;
  return SWA_OK;
}

}  // namespace

extern "C" swa_status_t swa_backward_noalloc(const swa_params_t* p, const void* q, const void* k, const void* v,
                                             const void* dy, const void* out, const float* softmax_max,
                                             const float* softmax_sum, const uint8_t* drop_mask, void* dq, void* dk,
                                             void* dv, swa_stream_t stream) {
  size_t need = 0;
  swa_status_t st = swa_backward_workspace_size(p, &need);
  if (st != SWA_OK) return st;
  if (need > kNoAllocScratchBytes)
    return swa::set_error(SWA_ERR_WORKSPACE,
                          "this problem needs %zu bytes of scratch; swa_backward_noalloc has a fixed %zu bytes "
                          "(64 MiB); use swa_backward with a workspace",
                          need, kNoAllocScratchBytes);
  void* scratch = nullptr;
  st = scratch_in_current_context(&scratch);
  if (st != SWA_OK) return st;
  return swa_backward(p, q, k, v, dy, out, softmax_max, softmax_sum, drop_mask, dq, dk, dv, scratch,
                      kNoAllocScratchBytes, stream);
}
