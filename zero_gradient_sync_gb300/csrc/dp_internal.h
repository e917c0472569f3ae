// Interface between the C ABI (dp_api.cu) and the kernel launchers (dp_kernels.cu).
#pragma once

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stdint.h>

#include "dp_device.cuh"
#include "dpstep.h"

namespace dp {

struct PlanSeg {
  int64_t goff, loff;
  int32_t tile0, owner;
};

// A validated layout, empty segments dropped, tiles counted.
struct Plan {
  int32_t n, stage, nseg, ntiles;
  int64_t psi;
  int64_t shard_len[DP_MAX_N];
  PlanSeg e[DP_MAX_SEG + 1];  // e[nseg] = {psi, 0, ntiles, 0}
};

struct StepScalars {
  float lr, beta1, beta2, eps, omb1, omb2;
  float inv;  // fl32(1 / (n S))
  int32_t mode;   // DP_SUM_COMPENSATED or DP_SUM_PLAIN
  int32_t order;  // DP_ORDER_RING or DP_ORDER_TREE
  uint64_t timeout_ns;
  ScalerK scaler;  // disabled unless the step uses the device-resident loss scale
  int32_t defer;   // DP_DEFER_COMMIT: the reduction publishes found_inf only; dp_commit_* commits later
};

// A named range on the host timeline around the launches of one phase of the step (pass A, pass B, ...), so a
// trace splits a step into its phases; costs nothing unless a profiler is attached (NVTX v3, header-only).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

// Records msg as this thread's dp_last_error() and returns s.
dp_status_t report_error(dp_status_t s, const char* msg);

// Each launcher returns the launch's cudaError_t and adds to *launches.
cudaError_t launch_reduce(const Plan& P, const uint16_t* const* g, int a, float* const* gbar, const StepScalars& s,
                          int advance, dp_step_state_t* st, cudaStream_t stream, uint64_t* launches);
// Tree order (dp_tree.cu): pass A and the staged reduce-scatter.
cudaError_t launch_reduce_tree(const Plan& P, const uint16_t* const* g, int a, float* const* gbar,
                               const StepScalars& s, int advance, dp_step_state_t* st, cudaStream_t stream,
                               uint64_t* launches);
cudaError_t launch_rs_tree(const Plan& P, const float* const* acc, float* const* gbar, const StepScalars& s,
                           dp_step_state_t* st, cudaStream_t stream, uint64_t* launches);
// Per-micro-step reduce-scatter (dp_micro.cu): micro-step k of a into the owner shard accumulators.
cudaError_t launch_rs_micro(const Plan& P, const uint16_t* const* g, float* const* acc, float* const* gbar, int k,
                            int a, const StepScalars& s, dp_step_state_t* st, cudaStream_t stream,
                            uint64_t* launches);
cudaError_t launch_single_pass(const Plan& P, const uint16_t* const* g, int a, uint16_t* const* rep,
                               float* const* master2, float* const* m2, float* const* v2, const StepScalars& s,
                               dp_step_state_t* st, cudaStream_t stream, uint64_t* launches);
cudaError_t launch_update(const Plan& P, uint16_t* const* rep, float* const* master, float* const* m,
                          float* const* v, const float* const* gbar, const StepScalars& s,
                          const dp_step_state_t* st, cudaStream_t stream, uint64_t* launches);
cudaError_t launch_accumulate(float* const* acc, const uint16_t* const* g, int64_t psi, int n, int first, int mode,
                              cudaStream_t stream, uint64_t* launches);
cudaError_t launch_rs_avg(const Plan& P, const float* const* acc, float* const* gbar, const StepScalars& s,
                          dp_step_state_t* st, cudaStream_t stream, uint64_t* launches);
cudaError_t launch_advance(dp_step_state_t* st, double b1, double b2, cudaStream_t stream, uint64_t* launches);
cudaError_t launch_allgather(const Plan& P, uint16_t* const* rep, const float* const* master,
                             const dp_step_state_t* st, cudaStream_t stream, uint64_t* launches);
cudaError_t launch_state_init(dp_step_state_t* st, cudaStream_t stream, uint64_t* launches);
// Deferred commit (one thread) and the single pass's replica repair (work only on a skipped step).
cudaError_t launch_commit(dp_step_state_t* st, double b1, double b2, const ScalerK& scaler, int flip_set,
                          cudaStream_t stream, uint64_t* launches);
cudaError_t launch_repair(const Plan& P, uint16_t* const* rep, float* const* master2, const dp_step_state_t* st,
                          cudaStream_t stream, uint64_t* launches);
cudaError_t launch_scaler_init(dp_step_state_t* st, float scale, cudaStream_t stream, uint64_t* launches);
cudaError_t launch_selftest_wait(dp_step_state_t* st, uint64_t timeout_ns, cudaStream_t stream, uint64_t* launches);

}  // namespace dp
