// Interface between the C ABI (dp_api.cu) and the kernel launchers (dp_kernels.cu).
#pragma once

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stdint.h>

#include <vector>

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
  std::vector<PlanSeg> e;  // nseg + 1 entries; e[nseg] = {end of the last segment, 0, ntiles, 0}
};

struct StepScalars {
  float lr, beta1, beta2, eps, omb1, omb2;
  float inv;  // fl32(1 / (n S))
  int32_t mode;   // DP_SUM_COMPENSATED or DP_SUM_PLAIN
  int32_t order;  // DP_ORDER_RING or DP_ORDER_TREE
  uint64_t timeout_ns;
  ScalerK scaler;  // disabled unless the step uses the device-resident loss scale
  int32_t defer;   // DP_DEFER_COMMIT: the reduction publishes found_inf only; dp_commit_* commits later
  int32_t merge;   // a later launch of one reduction: its finish ORs into found_inf and adds to nonfinite
};

// Segments one launch takes in its by-value table.  A layout with more segments runs as several launches over
// contiguous runs of at most this many segments -- contiguous ranges of the parameter space, whose elements
// keep their global and local indices.  Reductions then publish the skip decision over all the launches: the
// first launch's finish sets found_inf and nonfinite, later ones OR and add into them, and only the last one
// commits.
constexpr int KERNEL_SEG = DP_KERNEL_SEG;

// The plan of segments [s0, s1) of P, tiles renumbered from 0 (psi, n, stage and shard lengths kept).
inline void chunk_plan(const Plan& P, int s0, int s1, Plan& C) {
  C.n = P.n;
  C.stage = P.stage;
  C.psi = P.psi;
  for (int r = 0; r < DP_MAX_N; ++r) C.shard_len[r] = P.shard_len[r];
  C.nseg = s1 - s0;
  C.e.resize((size_t)C.nseg + 1);
  const int32_t t0 = P.e[s0].tile0;
  for (int k = s0; k <= s1; ++k) {
    C.e[k - s0] = P.e[k];
    C.e[k - s0].tile0 -= t0;
  }
  C.e[C.nseg].loff = 0;
  C.e[C.nseg].owner = 0;
  C.ntiles = C.e[C.nseg].tile0;
}

// f(plan, scalars, last) once for P itself, or once per chunk of at most KERNEL_SEG segments with the
// scalars of that launch (merge on every chunk but the first, defer on every chunk but the last).
template <typename F>
cudaError_t for_each_chunk(const Plan& P, const StepScalars& s, F&& f) {
  if (P.nseg <= KERNEL_SEG) return f(P, s, true);
  static thread_local Plan C;
  for (int s0 = 0; s0 < P.nseg; s0 += KERNEL_SEG) {
    const int s1 = P.nseg - s0 < KERNEL_SEG ? P.nseg : s0 + KERNEL_SEG;
    const bool last = s1 == P.nseg;
    chunk_plan(P, s0, s1, C);
    StepScalars sc = s;
    sc.merge = s0 > 0 ? 1 : 0;
    sc.defer = (s.defer || !last) ? 1 : 0;
    const cudaError_t e = f(static_cast<const Plan&>(C), static_cast<const StepScalars&>(sc), last);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

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
