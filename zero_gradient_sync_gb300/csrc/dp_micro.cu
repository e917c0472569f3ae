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
// One launch per micro-step.  One producer thread streams, per half tile, the owner's accumulator piece (its
// 16-byte-aligned interior in local space) and then the n ranks' bf16 gradient pieces in ring order, by 1-D
// bulk copies (cp.async.bulk, mbarrier transaction counts) into a ring of six 30 KB shared-memory slots; 15
// consumer warps own 8 elements a thread, take their accumulator values (the <= 1 (hi, lo) pair or <= 3 floats
// outside the copied interior from global memory), fold four gradient inputs a stage in ring order, add the
// micro-step's sum into the accumulator and write it back at the owner's local index with 16-byte stores where
// the local offset allows.  The last micro-step's launch writes gbar instead, counts non-finite values and
// publishes the skip decision and t like pass A of the step.  Every wait is bounded.
//
// With one micro-step (a = 1) the per-micro-step order is the step's own ring order, operation for
// operation: the same result as dp_step's pass A, which runs on the ring kernel.
#include <type_traits>

#include "dp_device.cuh"
#include "dp_internal.h"
#include "dp_launch.h"

namespace dp {
namespace {

// Launch shape: one producer warp whose lane 0 issues every bulk copy, and 15 consumer warps that own 8
// elements each, so a stage input is half a tile (3840 elements, 7.5 KB of bf16).  A stage carries either four
// gradient inputs (30 KB) or the owner's accumulator piece for the half tile (its 16-byte-aligned interior in
// local space: <= 30 KB of (hi, lo) pairs compensated, <= 15 KB plain), so every slot is 30 KB; six slots keep
// 180 KB in flight per SM.
constexpr int RM_CWARPS = 15;
constexpr int RM_CTHREADS = RM_CWARPS * 32;
constexpr int RM_THREADS = RM_CTHREADS + 32;
constexpr int RM_EPT = 8;
constexpr int RM_SUB = RM_CTHREADS * RM_EPT;       // elements of a half tile
constexpr int RM_IN_BYTES = RM_SUB * 2;            // one gradient input's half tile
constexpr int RM_NPS = 4;                          // gradient inputs per stage
constexpr int RM_SLOT = RM_NPS * RM_IN_BYTES;      // 30 KB: four inputs, or one accumulator piece
constexpr int RM_NST = 6;
constexpr int RM_SMEM = RM_NST * RM_SLOT + 2 * RM_NST * 8 + 32;
static_assert(TILE == 2 * RM_SUB, "a tile is two half tiles");
static_assert(RM_SUB * 8 <= RM_SLOT, "a half tile's (hi, lo) pairs fit one slot");
static_assert(RM_SMEM + 64 <= 227 * 1024, "shared memory fits one CTA");

enum { RM_FIRST = 1, RM_LAST = 2 };   // flags: no accumulator to read / write gbar and finish

template <int MAXSEG>
struct MicroParams {
  const uint16_t* g[DP_MAX_N];   // micro-step k of every rank
  float* acc[DP_MAX_N];          // owner shards: hi (plain) or interleaved (hi, lo) pairs (compensated)
  float* gbar[DP_MAX_N];
  dp_step_state_t* state;
  uint64_t timeout_ns;
  double beta1, beta2;
  float inv;
  int32_t n;
  int32_t advance;  // last launch: commit the step (0 when the commit is deferred)
  int32_t merge;    // a later launch of one reduction (see finish_reduction)
  ScalerK scaler;   // enabled (last launch only): unscale by the device-resident scale
  SegTable<MAXSEG> seg;
};

template <int NST>
struct MicroPos {
  uint32_t slot = 0, phase = 0, count = 0;
  __device__ __forceinline__ void next() {
    ++count;
    if (++slot == NST) {
      slot = 0;
      phase ^= 1u;
    }
  }
};

// Half h of tile t: its global range [lo, hi) and the 8-aligned start sa of the gradients' copy.
struct MicroHalf {
  int64_t lo, hi, sa;
};
__device__ __forceinline__ MicroHalf micro_half(const Tile& t, int h) {
  const int64_t cb = (t.start / TILE) * TILE + (int64_t)h * RM_SUB;
  MicroHalf x;
  x.lo = t.start > cb ? t.start : cb;
  x.hi = t.end < cb + RM_SUB ? t.end : cb + RM_SUB;
  x.sa = x.lo & ~int64_t(7);
  return x;
}

// The accumulator's bulk-copied interior [jlo, jhi) (local indices) of the local range [js, je): 16-byte
// aligned in the accumulator array (pairs of (hi, lo) compensated, groups of four plain).
template <bool COMP>
__device__ __forceinline__ void acc_interior(int64_t js, int64_t je, int64_t& jlo, int64_t& jhi) {
  constexpr int64_t al = COMP ? 2 : 4;
  jlo = (js + al - 1) & ~(al - 1);
  jhi = je & ~(al - 1);
  if (jhi < jlo) jhi = jlo;
}

template <int MAXSEG, bool COMP, int FLAGS>
__global__ void __launch_bounds__(RM_THREADS, 1) rs_micro_kernel(const __grid_constant__ MicroParams<MAXSEG> p) {
  constexpr bool FIRST = (FLAGS & RM_FIRST) != 0, LAST = (FLAGS & RM_LAST) != 0;
  extern __shared__ __align__(1024) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + RM_NST * RM_SLOT);
  uint64_t* empty = full + RM_NST;
  volatile int* s_abort = reinterpret_cast<volatile int*>(empty + RM_NST);
  unsigned long long* s_count = reinterpret_cast<unsigned long long*>(empty + RM_NST + 1);
  __shared__ float s_inv;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n = p.n;
  const int ntiles = p.seg.ntiles;
  const int64_t psi = p.seg.psi;
  const int64_t p8 = psi & ~int64_t(7);

  if (tid == 0) {
    for (int q = 0; q < RM_NST; ++q) {
      mbar_init(smem_u32(&full[q]), 1);
      mbar_init(smem_u32(&empty[q]), RM_CWARPS);
    }
    *s_abort = 0;
    *s_count = 0ull;
    float inv = p.inv;
    if (LAST && p.scaler.enabled) {
      // fl32(1 / (n S)) from the device-resident scale, as the host computes it for a fixed scale.
      const float sc = *reinterpret_cast<volatile const float*>(&p.state->loss_scale);
      inv = (float)(1.0 / ((double)p.n * (double)sc));
      if (!(sc > 0.0f) || nonfinite(sc) || !(inv >= 1.17549435e-38f) || nonfinite(inv)) {
        record_error(p.state, DP_ERR_INVALID_ARG);
        *s_abort = 1;    // skip the work; the finish sees the error and skips the step
        inv = 0.0f;
      }
    }
    s_inv = inv;
    fence_mbar_init();
  }
  __syncthreads();
  // A bad device scale skips every tile, in every thread alike.
  const int tile0 = *s_abort ? ntiles : (int)blockIdx.x;

  unsigned bad = 0;
  if (warp == RM_CWARPS) {
    // ------------------------------------------------------------ producer: accumulator piece, then the ranks
    if (lane == 0) {
      MicroPos<RM_NST> sp;
      TileWalker<MAXSEG> walk;
      auto acquire = [&]() {
        if (sp.count >= (uint32_t)RM_NST &&
            !mbar_wait_bounded(smem_u32(&empty[sp.slot]), sp.phase ^ 1u, p.timeout_ns, s_abort)) {
          if (!*s_abort) record_error(p.state, DP_ERR_TIMEOUT);
          *s_abort = 1;
          return false;
        }
        return true;
      };
      for (int tile = tile0; tile < ntiles && !*s_abort; tile += gridDim.x) {
        const Tile t = walk.at(p.seg, tile);
        const int64_t delta = t.loff - t.goff;
        for (int h = 0; h < 2 && !*s_abort; ++h) {
          const MicroHalf x = micro_half(t, h);
          if (x.lo >= x.hi) continue;
          if (!FIRST) {
            if (!acquire()) break;
            int64_t jlo, jhi;
            acc_interior<COMP>(x.lo + delta, x.hi + delta, jlo, jhi);
            const uint32_t bytes = (uint32_t)(jhi - jlo) * (COMP ? 8u : 4u);
            const uint32_t fb = smem_u32(&full[sp.slot]);
            mbar_arrive_expect_tx(fb, bytes);
            if (bytes) bulk_g2s(smem_u32(smem + sp.slot * RM_SLOT), p.acc[t.owner] + (COMP ? 2 : 1) * jlo, bytes, fb);
            sp.next();
          }
          int64_t sb = (x.hi + 7) & ~int64_t(7);
          if (sb > p8) sb = p8;
          const uint32_t bytes = sb > x.sa ? (uint32_t)(sb - x.sa) * 2u : 0u;
          // Ranks in ring order: owner + 1 first, the owner last; four to a stage.
          int r = t.owner + 1 == n ? 0 : t.owner + 1;
          for (int q = 0; q < n && !*s_abort; q += RM_NPS) {
            if (!acquire()) break;
            const int cnt = n - q < RM_NPS ? n - q : RM_NPS;
            const uint32_t fb = smem_u32(&full[sp.slot]);
            mbar_arrive_expect_tx(fb, bytes * (uint32_t)cnt);
            for (int hh = 0; hh < cnt; ++hh) {
              if (bytes) bulk_g2s(smem_u32(smem + sp.slot * RM_SLOT + hh * RM_IN_BYTES), p.g[r] + x.sa, bytes, fb);
              if (++r == n) r = 0;
            }
            sp.next();
          }
        }
      }
      // Never leave with copies in flight: wait for the newest issued phase of every slot.
      if (*s_abort) {
        const uint32_t it = sp.count;
        const uint32_t first = it > (uint32_t)RM_NST ? it - RM_NST : 0u;
        for (uint32_t y = first; y < it; ++y)
          (void)mbar_wait_bounded(smem_u32(&full[y % RM_NST]), (y / RM_NST) & 1u, p.timeout_ns, nullptr);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ consumers: 8 elements per thread
    const float inv = s_inv;
    MicroPos<RM_NST> sp;
    TileWalker<MAXSEG> walk;
    bool live = true;
    auto wait_full = [&]() {
      if (live && !mbar_wait_bounded(smem_u32(&full[sp.slot]), sp.phase, p.timeout_ns, s_abort)) {
        if (!*s_abort) record_error(p.state, DP_ERR_TIMEOUT);
        *s_abort = 1;
        live = false;
      }
    };
    // The slot is refilled by the async proxy (bulk copy): order this thread's reads of it before that write.
    auto release = [&]() {
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty[sp.slot]));
      sp.next();
    };
    const f2_t inv2 = f2_pack(inv, inv);
    for (int tile = tile0; tile < ntiles; tile += gridDim.x) {
      const Tile t = walk.at(p.seg, tile);
      const int64_t delta = t.loff - t.goff;
      float* accp = p.acc[t.owner];
      for (int h = 0; h < 2; ++h) {
        const MicroHalf x = micro_half(t, h);
        if (x.lo >= x.hi) continue;
        // WHOLE: the half tile is a whole half cell below the buffer's last partial 8-group, so every thread
        // holds 8 elements of it and every gradient value is in shared memory: no guards.
        auto body = [&](auto whole_tag) {
          constexpr bool WHOLE = decltype(whole_tag)::value;
          const int64_t e0 = x.sa + RM_EPT * tid;
          const bool active = WHOLE || e0 < x.hi;
          const bool tailgrp = !WHOLE && active && (e0 + RM_EPT > p8);
          const int64_t j = e0 + delta;   // local index of element e0 (only elements inside the half are used)

          // The owner's accumulator for these 8 elements as packed pairs: hi AH[u] and (compensated) lo AL[u]
          // of elements 2u, 2u + 1.  From the copied interior; its ragged ends from global memory.
          f2_t AH[4], AL[4];
          if (!FIRST) {
            wait_full();
            int64_t jlo, jhi;
            acc_interior<COMP>(x.lo + delta, x.hi + delta, jlo, jhi);
            const float* sa = reinterpret_cast<const float*>(smem + sp.slot * RM_SLOT);
            if (WHOLE && jlo == x.lo + delta && jhi == x.hi + delta) {
              // The interior is the whole half: this thread's values start at pair / float 8 * tid.
              if (COMP) {
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                  const float4 v = reinterpret_cast<const float4*>(sa)[4 * tid + u];
                  AH[u] = f2_pack(v.x, v.z);
                  AL[u] = f2_pack(v.y, v.w);
                }
              } else {
                const float4 v0 = reinterpret_cast<const float4*>(sa)[2 * tid];
                const float4 v1 = reinterpret_cast<const float4*>(sa)[2 * tid + 1];
                AH[0] = f2_pack(v0.x, v0.y); AH[1] = f2_pack(v0.z, v0.w);
                AH[2] = f2_pack(v1.x, v1.y); AH[3] = f2_pack(v1.z, v1.w);
              }
            } else {
              float ah[RM_EPT], al[RM_EPT];
#pragma unroll
              for (int u = 0; u < RM_EPT; ++u) {
                ah[u] = al[u] = 0.0f;
                const int64_t ju = j + u;
                if (active && live && e0 + u >= x.lo && e0 + u < x.hi) {
                  if (ju >= jlo && ju < jhi) {
                    if (COMP) {
                      const float2 v = *reinterpret_cast<const float2*>(sa + 2 * (ju - jlo));
                      ah[u] = v.x;
                      al[u] = v.y;
                    } else {
                      ah[u] = sa[ju - jlo];
                    }
                  } else {
                    ah[u] = COMP ? accp[2 * ju] : accp[ju];
                    if (COMP) al[u] = accp[2 * ju + 1];
                  }
                }
              }
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                AH[u] = f2_pack(ah[2 * u], ah[2 * u + 1]);
                AL[u] = f2_pack(al[2 * u], al[2 * u + 1]);
              }
            }
            release();
          }

          // p_k for these 8 elements: the ranks in ring order (input q is rank owner + 1 + q), four a stage.
          f2_t H[4], L[4];
          auto input = [&](const unsigned char* src_s, int q) -> uint4 {
            if (WHOLE) return *reinterpret_cast<const uint4*>(src_s);
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (active && live) {
              if (!tailgrp) {
                v = *reinterpret_cast<const uint4*>(src_s);
              } else {
                int rr = t.owner + 1 + q;
                while (rr >= n) rr -= n;
                const uint16_t* src = p.g[rr];
                uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
                for (int u = 0; u < RM_EPT; ++u) {
                  const uint32_t bb = (e0 + u < psi) ? (uint32_t)src[e0 + u] : 0u;
                  w[u >> 1] |= (u & 1) ? (bb << 16) : bb;
                }
                v = make_uint4(w[0], w[1], w[2], w[3]);
              }
            }
            return v;
          };
          auto fold = [&](const uint4& v) {
            const uint32_t ww[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const f2_t xx = bf16x2_to_f2(ww[u]);
              if (COMP) {
                f2_t e;
                H[u] = f2_two_sum(H[u], xx, e);
                L[u] = f2_add(L[u], e);
              } else {
                H[u] = f2_add(H[u], xx);
              }
            }
          };
          for (int q = 0; q < n; q += RM_NPS) {
            const int cnt = n - q < RM_NPS ? n - q : RM_NPS;
            wait_full();
            const unsigned char* src_s = smem + sp.slot * RM_SLOT + 2 * RM_EPT * tid;
            int hh = 0;
            if (q == 0) {   // the chain's first input
              const uint4 v = input(src_s, 0);
              const uint32_t ww[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                H[u] = bf16x2_to_f2(ww[u]);
                L[u] = 0ull;
              }
              hh = 1;
            }
            if (WHOLE && cnt == RM_NPS) {   // inputs in order: input 0 (unless it started the chain), then 1..3
              if (hh == 0) fold(input(src_s, q));
#pragma unroll
              for (int u = 1; u < RM_NPS; ++u) fold(input(src_s + u * RM_IN_BYTES, q + u));
            } else {
              for (; hh < cnt; ++hh) fold(input(src_s + hh * RM_IN_BYTES, q + hh));
            }
            release();
          }
          if (!active) return;

          if (!FIRST) {
            // A += p:  (H, e) = TwoSum(A_H, p_H), A_L = (A_L + e) + p_L  (plain: A = A + p)
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              if (COMP) {
                f2_t e;
                const f2_t s2 = f2_two_sum(AH[u], H[u], e);
                L[u] = f2_add(f2_add(AL[u], e), L[u]);
                H[u] = s2;
              } else {
                H[u] = f2_add(AH[u], H[u]);
              }
            }
          }
          const bool whole = WHOLE || (e0 >= x.lo && e0 + RM_EPT <= x.hi);
          if (!LAST) {
            float hv[RM_EPT], lv[RM_EPT];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              f2_unpack(H[u], hv[2 * u], hv[2 * u + 1]);
              if (COMP) f2_unpack(L[u], lv[2 * u], lv[2 * u + 1]);
            }
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
                if (e0 + u >= x.lo && e0 + u < x.hi) {
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
            for (int u = 0; u < 4; ++u) f2_unpack(f2_mul(COMP ? f2_add(H[u], L[u]) : H[u], inv2), o[2 * u], o[2 * u + 1]);
            float* dst = p.gbar[t.owner] + j;
            if (whole && ((reinterpret_cast<uintptr_t>(dst) & 15) == 0)) {
              *reinterpret_cast<float4*>(dst) = make_float4(o[0], o[1], o[2], o[3]);
              *reinterpret_cast<float4*>(dst + 4) = make_float4(o[4], o[5], o[6], o[7]);
#pragma unroll
              for (int u = 0; u < RM_EPT; ++u) bad += nonfinite(o[u]);
            } else {
#pragma unroll
              for (int u = 0; u < RM_EPT; ++u)
                if (e0 + u >= x.lo && e0 + u < x.hi) {
                  dst[u] = o[u];
                  bad += nonfinite(o[u]);
                }
            }
          }
        };
        if (x.hi - x.lo == RM_SUB && x.hi <= p8) body(std::true_type{});
        else body(std::false_type{});
      }
    }
  }

  if (LAST) {
    unsigned long long c = bad;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) c += __shfl_xor_sync(0xFFFFFFFFu, c, off);
    __syncthreads();
    if (lane == 0 && c) atomicAdd(s_count, c);
    __syncthreads();
    if (tid == 0)
      finish_reduction(p.state, *s_count, (*s_count != 0ull) || *s_abort, p.advance, p.beta1, p.beta2, &p.scaler,
                       0, p.merge);
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
  prm.timeout_ns = s.timeout_ns;
  prm.beta1 = (double)s.beta1;
  prm.beta2 = (double)s.beta2;
  prm.inv = s.inv;
  prm.n = P.n;
  prm.advance = s.defer ? 0 : 1;
  prm.merge = s.merge;
  prm.scaler = s.scaler;
  fill_seg(prm.seg, P);
  auto kern = rs_micro_kernel<MAXSEG, COMP, FLAGS>;
  // The opt-in shared-memory size is set once per device (not inside a stream capture on later calls).
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, RM_SMEM);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  // One CTA per SM over the tiles; every CTA of the last launch joins the grid-wide finish, so at least one.
  int grid = sm_count();
  if (P.ntiles < grid) grid = P.ntiles > 0 ? P.ntiles : 1;
  kern<<<grid, RM_THREADS, RM_SMEM, stream>>>(prm);
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

cudaError_t launch_rs_micro(const Plan& P0, const uint16_t* const* g, float* const* acc, float* const* gbar, int k,
                            int a, const StepScalars& s0, dp_step_state_t* st, cudaStream_t stream,
                            uint64_t* launches) {
  return for_each_chunk(P0, s0, [&](const Plan& P, const StepScalars& s, bool) {
    ++*launches;
    const bool comp = s.mode == DP_SUM_COMPENSATED;
    if (P.nseg <= SMALL_SEG)
      return comp ? launch_micro_c<SMALL_SEG, true>(P, g, acc, gbar, k, a, s, st, stream)
                  : launch_micro_c<SMALL_SEG, false>(P, g, acc, gbar, k, a, s, st, stream);
    return comp ? launch_micro_c<BIG_SEG, true>(P, g, acc, gbar, k, a, s, st, stream)
                : launch_micro_c<BIG_SEG, false>(P, g, acc, gbar, k, a, s, st, stream);
  });
}

}  // namespace dp
