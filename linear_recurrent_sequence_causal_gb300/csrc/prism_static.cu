// prism_forward_static: the full forward pass with a scratch area that lives in
// this library's own device memory instead of a caller-provided workspace.
//
// Who needs it: callers that cannot allocate device memory at the point where
// they run the layer, e.g. code running inside a pre-planned memory arena or a
// host framework that forbids allocation on its hot path, or plugins handed
// only input and output buffers.  They pass inputs and outputs as usual; the
// scratch comes from a fixed file-scope array.
//
// The array is PRISM_STATIC_SCRATCH_BYTES long and is held by every GPU that
// loads this library, for the life of the process.  All calls on a device
// share it and it keeps the last call's contents, so calls whose execution
// overlaps on the GPU (different streams, or different host threads without
// ordering) race on it and must be serialised by the caller.
#include <cuda_runtime.h>

#include "../../include/prism.h"

namespace {

static __device__ __align__(256) unsigned char g_scratch[PRISM_STATIC_SCRATCH_BYTES];

// Device address of g_scratch on the current device, looked up on every call with
// that device current.  In host code g_scratch only names a host-side stand-in, so
// the address must come from the runtime; it is not cached, because the module can
// be loaded again at another address (after cudaDeviceReset, or in another context
// on the same device) and a stale address would send the kernels to memory this
// library no longer owns.  Once the module is loaded the lookup is a table read.
int scratch_for_current_device(void** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return PRISM_ERR_CUDA;
  *out = p;
  return PRISM_OK;
}

}  // namespace

extern "C" PRISM_API int prism_forward_static(const prism_dims* dims, const void* q, const void* k,
                                              const void* v, const float* log_alpha,
                                              const float* beta, const float* conv_w,
                                              const float* Wk, const float* Wp, const float* wbeta,
                                              float* out, float* final_state,
                                              const int32_t* seq_lens, void* stream) {
  size_t offsets[PRISM_WS_COUNT];
  const int check = prism_workspace_layout(dims, offsets, PRISM_WS_COUNT);   // validates dims
  if (check != PRISM_OK) return check;
  if (prism_workspace_bytes(dims) > (size_t)PRISM_STATIC_SCRATCH_BYTES) return PRISM_ERR_SCRATCH_LIMIT;
  void* ws = nullptr;
  const int rc = scratch_for_current_device(&ws);
  if (rc != PRISM_OK) return rc;
  // prism_forward clears the status words it needs; every other region is
  // written before it is read, so stale contents of a previous call are harmless.
  return prism_forward(dims, q, k, v, log_alpha, beta, conv_w, Wk, Wp, wbeta, out, final_state,
                       seq_lens, ws, (size_t)PRISM_STATIC_SCRATCH_BYTES, stream);
}

extern "C" PRISM_API int prism_static_status(const prism_dims* dims, int* status, void* stream) {
  size_t offsets[PRISM_WS_COUNT];
  const int check = prism_workspace_layout(dims, offsets, PRISM_WS_COUNT);   // validates dims
  if (check != PRISM_OK) return check;
  if (!status) return PRISM_ERR_INVALID_ARG;
  if (prism_workspace_bytes(dims) > (size_t)PRISM_STATIC_SCRATCH_BYTES) return PRISM_ERR_SCRATCH_LIMIT;
  void* ws = nullptr;
  const int rc = scratch_for_current_device(&ws);
  if (rc != PRISM_OK) return rc;
  return prism_device_status(dims, ws, (size_t)PRISM_STATIC_SCRATCH_BYTES, status, stream);
}
