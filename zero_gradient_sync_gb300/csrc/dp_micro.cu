// Per-micro-step reduce-scatter (sm_103a): the memory-saving form of ZeRO-2, where each micro-step's
// gradients are reduce-scattered as soon as they exist and summed into the owner's shard accumulator, so no
// rank keeps a full-length gradient accumulator ("Distributed Training: Split along the Four Axes", ZeRO /
// FSDP paragraph: stage 2 shards the gradients as well; "Data vs Tensor vs Pipeline Parallelism", sharded
// data parallelism: a reduce-scatter leaves each rank the sum of its own shard).
//
// Order for an element owned by s: p_k = g_{s+1,k} + g_{s+2,k} + ... + g_{s,k} (the ring's hops, one
// micro-step at a time), then A = ((p_0 + p_1) + ...) + p_{a-1}; gbar = fl32(A * fl32(1 / (n S))).
// Compensated: each p_k carries its TwoSum errors in a lo part (its first term has none), and the
// accumulator adds p_k as (H, e) = TwoSum(A_H, p_H), A_L = (A_L + e) + p_L; gbar uses A_H + A_L.
//
// One launch per micro-step, streaming its n bf16 inputs once with 16-byte loads (8 elements a thread,
// ranks in batches of eight, issued together with the accumulator's loads) and reading / writing the
// accumulator at the owner's local index.  The last micro-step's launch writes gbar instead, counts
// non-finite values and publishes the skip decision and t like pass A of the step.
//
// With one micro-step (a = 1) the per-micro-step order is the step's own ring order, operation for
// operation: the same result as dp_step's pass A, which runs on the ring kernel.
#include "dp_device.cuh"
#include "dp_internal.h"
#include "dp_launch.h"

namespace dp {
namespace {

constexpr int RM_THREADS = 256;
constexpr int RM_EPT = 8;
constexpr int RM_BATCH = 8;   // ranks whose loads are issued together

enum { RM_FIRST = 1, RM_LAST = 2 };   // flags: no accumulator to read / write gbar and finish

template <int MAXSEG>
struct MicroParams {
  const uint16_t* g[DP_MAX_N];   // micro-step k of every rank
  float* acc[DP_MAX_N];          // owner shards: hi (plain) or interleaved (hi, lo) pairs (compensated)
  float* gbar[DP_MAX_N];
  dp_step_state_t* state;
  double beta1, beta2;
  float inv;
  int32_t n;
  int32_t advance;  // last launch: commit the step (0 when the commit is deferred)
  ScalerK scaler;   // enabled (last launch only): unscale by the device-resident scale
  SegTable<MAXSEG> seg;
};

__device__ __forceinline__ uint4 load_group(const uint16_t* src, int64_t e0, int64_t psi) {
  if (e0 + RM_EPT <= psi) return __ldcs(reinterpret_cast<const uint4*>(src + e0));
  uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int u = 0; u < RM_EPT; ++u)
    if (e0 + u < psi) w[u >> 1] |= (uint32_t)src[e0 + u] << (16 * (u & 1));
  return make_uint4(w[0], w[1], w[2], w[3]);
}

template <int MAXSEG, bool COMP, int FLAGS>
__global__ void __launch_bounds__(RM_THREADS, 3) rs_micro_kernel(const __grid_constant__ MicroParams<MAXSEG> p) {
  constexpr bool FIRST = (FLAGS & RM_FIRST) != 0, LAST = (FLAGS & RM_LAST) != 0;
  __shared__ unsigned long long s_count;
  __shared__ float s_inv;
  __shared__ int s_bad_scale;
  if (LAST && threadIdx.x == 0) {
    s_count = 0ull;
    float inv = p.inv;
    int bad_scale = 0;
    if (p.scaler.enabled) {
      // fl32(1 / (n S)) from the device-resident scale, as the host computes it for a fixed scale.
      const float sc = *reinterpret_cast<volatile const float*>(&p.state->loss_scale);
      inv = (float)(1.0 / ((double)p.n * (double)sc));
      if (!(sc > 0.0f) || nonfinite(sc) || !(inv >= 1.17549435e-38f) || nonfinite(inv)) {
        record_error(p.state, DP_ERR_INVALID_ARG);
        bad_scale = 1;    // skip the work; the finish sees the error and skips the step
        inv = 0.0f;
      }
    }
    s_inv = inv;
    s_bad_scale = bad_scale;
  }
  if (LAST) __syncthreads();
  const float inv = LAST ? s_inv : 0.0f;
  const int n = p.n;
  const int64_t psi = p.seg.psi;
  unsigned bad = 0;
  TileWalker<MAXSEG> walk;
  for (int tile = (LAST && s_bad_scale) ? p.seg.ntiles : blockIdx.x; tile < p.seg.ntiles; tile += gridDim.x) {
    const Tile t = walk.at(p.seg, tile);
    const int64_t A = t.start & ~int64_t(7), B = (t.end + 7) & ~int64_t(7);
    const int64_t delta = t.loff - t.goff;
    for (int64_t e0 = A + RM_EPT * (int64_t)threadIdx.x; e0 < B; e0 += RM_EPT * RM_THREADS) {
      // The shard accumulator at the owner's local index: the group's elements inside the tile.  Its loads
      // are issued first, so they are in flight together with the gradients'.
      const bool whole = e0 >= t.start && e0 + RM_EPT <= t.end;
      float* accp = p.acc[t.owner];
      const int64_t j = delta + e0;   // local index of element e0 (only elements inside the tile are touched)
      float ah[RM_EPT], al[RM_EPT];
      if (!FIRST) {
        const bool vec = whole && (((reinterpret_cast<uintptr_t>(accp + (COMP ? 2 * j : j))) & 15) == 0);
        if (vec) {
          if (COMP) {
#pragma unroll
            for (int q = 0; q < RM_EPT / 2; ++q) {
              const float4 v = *reinterpret_cast<const float4*>(accp + 2 * (j + 2 * q));
              ah[2 * q] = v.x; al[2 * q] = v.y; ah[2 * q + 1] = v.z; al[2 * q + 1] = v.w;
            }
          } else {
#pragma unroll
            for (int q = 0; q < RM_EPT / 4; ++q) {
              const float4 v = *reinterpret_cast<const float4*>(accp + j + 4 * q);
              ah[4 * q] = v.x; ah[4 * q + 1] = v.y; ah[4 * q + 2] = v.z; ah[4 * q + 3] = v.w;
            }
          }
        } else {
#pragma unroll
          for (int u = 0; u < RM_EPT; ++u) {
            ah[u] = al[u] = 0.0f;
            if (e0 + u >= t.start && e0 + u < t.end) {
              ah[u] = COMP ? accp[2 * (j + u)] : accp[j + u];
              if (COMP) al[u] = accp[2 * (j + u) + 1];
            }
          }
        }
      }
      // p_k for these 8 elements: the ranks in ring order s+1, ..., s.
      f2_t H[4], L[4];
      int r = t.owner + 1 == n ? 0 : t.owner + 1;
      for (int j0 = 0; j0 < n; j0 += RM_BATCH) {
        uint4 w[RM_BATCH];
        int rr = r;
#pragma unroll
        for (int b = 0; b < RM_BATCH; ++b) {
          if (j0 + b < n) {
            w[b] = load_group(p.g[rr], e0, psi);
            if (++rr == n) rr = 0;
          }
        }
#pragma unroll
        for (int b = 0; b < RM_BATCH; ++b) {
          if (j0 + b < n) {
            const uint32_t ww[4] = {w[b].x, w[b].y, w[b].z, w[b].w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const f2_t x = bf16x2_to_f2(ww[u]);
              if (j0 + b == 0) {
                H[u] = x;
                L[u] = 0ull;
              } else if (COMP) {
                f2_t e;
                H[u] = f2_two_sum(H[u], x, e);
                L[u] = f2_add(L[u], e);
              } else {
                H[u] = f2_add(H[u], x);
              }
            }
          }
        }
        r = rr;
      }
      float hv[RM_EPT], lv[RM_EPT];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        f2_unpack(H[u], hv[2 * u], hv[2 * u + 1]);
        if (COMP) f2_unpack(L[u], lv[2 * u], lv[2 * u + 1]);
      }
      if (!FIRST) {
        // A += p
#pragma unroll
        for (int u = 0; u < RM_EPT; ++u) {
          if (COMP) {
            float err;
            const float s = two_sum(ah[u], hv[u], err);
            lv[u] = __fadd_rn(__fadd_rn(al[u], err), lv[u]);
            hv[u] = s;
          } else {
            hv[u] = __fadd_rn(ah[u], hv[u]);
          }
        }
      }
      if (!LAST) {
        const bool vec = whole && (((reinterpret_cast<uintptr_t>(accp + (COMP ? 2 * j : j))) & 15) == 0);
        if (vec) {
          if (COMP) {
#pragma unroll
            for (int q = 0; q < RM_EPT / 2; ++q)
              *reinterpret_cast<float4*>(accp + 2 * (j + 2 * q)) =
                  make_float4(hv[2 * q], lv[2 * q], hv[2 * q + 1], lv[2 * q + 1]);
          } else {
#pragma unroll
            for (int q = 0; q < RM_EPT / 4; ++q)
              *reinterpret_cast<float4*>(accp + j + 4 * q) =
                  make_float4(hv[4 * q], hv[4 * q + 1], hv[4 * q + 2], hv[4 * q + 3]);
          }
        } else {
#pragma unroll
          for (int u = 0; u < RM_EPT; ++u) {
            if (e0 + u >= t.start && e0 + u < t.end) {
              if (COMP) {
                accp[2 * (j + u)] = hv[u];
                accp[2 * (j + u) + 1] = lv[u];
              } else {
                accp[j + u] = hv[u];
              }
            }
          }
        }
      } else {
        float o[RM_EPT];
#pragma unroll
        for (int u = 0; u < RM_EPT; ++u) o[u] = __fmul_rn(COMP ? __fadd_rn(hv[u], lv[u]) : hv[u], inv);
        float* dst = p.gbar[t.owner] + j;
        if (whole && ((reinterpret_cast<uintptr_t>(dst) & 15) == 0)) {
          *reinterpret_cast<float4*>(dst) = make_float4(o[0], o[1], o[2], o[3]);
          *reinterpret_cast<float4*>(dst + 4) = make_float4(o[4], o[5], o[6], o[7]);
#pragma unroll
          for (int u = 0; u < RM_EPT; ++u) bad += nonfinite(o[u]);
        } else {
#pragma unroll
          for (int u = 0; u < RM_EPT; ++u)
            if (e0 + u >= t.start && e0 + u < t.end) {
              dst[u] = o[u];
              bad += nonfinite(o[u]);
            }
        }
      }
    }
  }
  if (LAST) {
    unsigned long long c = bad;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) c += __shfl_xor_sync(0xFFFFFFFFu, c, off);
    if ((threadIdx.x & 31) == 0 && c) atomicAdd(&s_count, c);
    __syncthreads();
    if (threadIdx.x == 0)
      finish_reduction(p.state, s_count, (s_count != 0ull) || s_bad_scale, p.advance, p.beta1, p.beta2, &p.scaler,
                       0);
  }
}

template <int MAXSEG, bool COMP, int FLAGS>
cudaError_t launch_micro_t(const Plan& P, const uint16_t* const* g, float* const* acc, float* const* gbar,
                           const StepScalars& s, dp_step_state_t* st, cudaStream_t stream) {
  MicroParams<MAXSEG> prm;
  for (int r = 0; r < P.n; ++r) {
    prm.g[r] = g[r];
    prm.acc[r] = acc ? acc[r] : nullptr;
    prm.gbar[r] = gbar ? gbar[r] : nullptr;
  }
  prm.state = st;
  prm.beta1 = (double)s.beta1;
  prm.beta2 = (double)s.beta2;
  prm.inv = s.inv;
  prm.n = P.n;
  prm.advance = s.defer ? 0 : 1;
  prm.scaler = s.scaler;
  fill_seg(prm.seg, P);
  auto kern = rs_micro_kernel<MAXSEG, COMP, FLAGS>;
  kern<<<occupancy_grid(kern, RM_THREADS, 0, P.ntiles), RM_THREADS, 0, stream>>>(prm);
  return cudaGetLastError();
}

template <int MAXSEG, bool COMP>
cudaError_t launch_micro_c(const Plan& P, const uint16_t* const* g, float* const* acc, float* const* gbar, int k,
                           int a, const StepScalars& s, dp_step_state_t* st, cudaStream_t stream) {
  const bool first = k == 0, last = k == a - 1;
  if (first && last) return launch_micro_t<MAXSEG, COMP, RM_FIRST | RM_LAST>(P, g, acc, gbar, s, st, stream);
  if (first) return launch_micro_t<MAXSEG, COMP, RM_FIRST>(P, g, acc, gbar, s, st, stream);
  if (last) return launch_micro_t<MAXSEG, COMP, RM_LAST>(P, g, acc, gbar, s, st, stream);
  return launch_micro_t<MAXSEG, COMP, 0>(P, g, acc, gbar, s, st, stream);
}

}  // namespace

cudaError_t launch_rs_micro(const Plan& P, const uint16_t* const* g, float* const* acc, float* const* gbar, int k,
                            int a, const StepScalars& s, dp_step_state_t* st, cudaStream_t stream,
                            uint64_t* launches) {
  ++*launches;
  const bool comp = s.mode == DP_SUM_COMPENSATED;
  if (P.nseg <= SMALL_SEG)
    return comp ? launch_micro_c<SMALL_SEG, true>(P, g, acc, gbar, k, a, s, st, stream)
                : launch_micro_c<SMALL_SEG, false>(P, g, acc, gbar, k, a, s, st, stream);
  return comp ? launch_micro_c<BIG_SEG, true>(P, g, acc, gbar, k, a, s, st, stream)
              : launch_micro_c<BIG_SEG, false>(P, g, acc, gbar, k, a, s, st, stream);
}

}  // namespace dp
