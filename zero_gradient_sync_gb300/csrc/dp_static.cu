// dp_step_static: the fused step for callers that cannot allocate device memory.
//
// dp_step needs scratch space for the averaged-gradient shards between its
// two kernels, and expects the caller to allocate it.  Some callers cannot:
// a plugin inside a host runtime that owns every device allocation and plans
// its memory once at start-up, a real-time loop that must not allocate
// after initialisation, or code that runs while another allocator holds a
// lock it would need.  This entry point keeps that scratch in a fixed array
// compiled into the library instead, so the caller passes only inputs and
// outputs and nothing is allocated on any call.
//
// The array is DP_STATIC_SCRATCH_BYTES (64 MiB) per GPU and stays reserved
// on every device that loads the library until the process exits.  All calls
// share it: two calls whose kernels overlap on the GPU (on different streams,
// or on one stream from different threads without ordering) race on it.
// Nothing in it has to start at zero -- the reduce kernel writes every
// scratch element it later reads -- so it is never cleared.
#include <cstdio>

#include "dp_device.cuh"
#include "dp_internal.h"
#include "dpstep.h"

static_assert(DP_STATIC_SCRATCH_BYTES % 256 == 0, "scratch size must keep 256-byte shard alignment");

static __device__ __align__(256) unsigned char g_static_scratch[DP_STATIC_SCRATCH_BYTES];

namespace {

// Device address of g_static_scratch in the context current on this thread.  In host code the symbol itself
// only names a host-side shadow, never the device memory, so every call asks the runtime for the address:
// the lookup is cheap, and a cached address would go stale when the context changes under the same device
// number (a cudaDeviceReset, or another context made current on the device).
cudaError_t scratch_address(void** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
  if (e != cudaSuccess) return e;
  *out = p;
  return cudaSuccess;
}

}  // namespace

extern "C" dp_status_t dp_step_static(uint16_t* const* replicas, float* const* master, float* const* m,
                                      float* const* v, const uint16_t* const* grads, int32_t a,
                                      const dp_layout_t* layout, dp_adam_t adam, float loss_scale,
                                      int32_t sum_mode, dp_step_state_t* d_state, dp_stream_t stream) {
  // Size check first: the shards must fit the fixed array, each 256-byte aligned.
  const size_t need = dp_workspace_size(layout);
  if (need == 0) return dp_layout_validate(layout);   // invalid layout: report its error
  if (need > (size_t)DP_STATIC_SCRATCH_BYTES) {
    char msg[256];
    snprintf(msg, sizeof(msg),
             "dp_step_static: the gradient shards need %zu bytes, more than the %lld-byte static scratch", need,
             (long long)DP_STATIC_SCRATCH_BYTES);
    return dp::report_error(DP_ERR_INVALID_ARG, msg);
  }
  void* ws = nullptr;
  const cudaError_t e = scratch_address(&ws);
  if (e != cudaSuccess) {
    char msg[256];
    snprintf(msg, sizeof(msg), "dp_step_static: cudaGetSymbolAddress failed: %s", cudaGetErrorString(e));
    return dp::report_error(DP_ERR_CUDA, msg);
  }
  // The same two kernels as dp_step, with the shards carved out of the static array.
  return dp_step(replicas, master, m, v, grads, a, layout, adam, loss_scale, sum_mode, nullptr, ws, d_state,
                 stream);
}
