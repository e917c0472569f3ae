// Kernels of the fused data-parallel step and their launchers (sm_103a).
//
// reduce (fused pass A): the n*a bf16 micro-step gradients of a tile are
//   streamed once from HBM into a ring of shared-memory stages (two inputs,
//   two 15 KB bulk copies, per stage) by one producer thread issuing 1-D
//   bulk copies (cp.async.bulk, mbarrier transaction counts); 15 consumer
//   warps fold each stage into per-element accumulators in the fixed ring
//   order (ranks s+1..s, each rank's micro-steps 0..a-1), scale by
//   fl32(1/(n S)), count non-finite results and write gbar to the owner's
//   shard.  The last CTA publishes the step's skip flag and advances t.
// update (fused pass B): unless skipped, Adam on the fp32 master/m/v shard
//   (16-byte vector loads/stores in local index space) and the bf16 image of
//   the new master staged in shared memory, then bulk-stored into all n
//   replicas (cp.async.bulk shared->global) at global index.
// single pass (reduce with FUSED != 0): pass A's stream, then each tile's
//   update from gbar on chip and the tile's old optimizer state, bulk-copied
//   into shared memory while its gradients stream, into the other of two
//   state sets (made current by the last CTA unless skipped); repair rewrites
//   the replicas on a skipped step.
// update, plain data parallelism (stage 0): every rank's full-length state
//   updated with the owner's gbar, 16-byte vectors over (rank, 4-group) items.
// Staged kernels (accumulate, rs_avg, adam = update without replicas,
//   allgather, advance) compute the same step one phase at a time: bit-
//   identical in plain arithmetic; compensated, the staged form keeps one
//   (hi, lo) pair per rank where pass A carries one pair through all inputs.
// commit: the step state's commit for a reduction that deferred it.
#include <algorithm>
#include <type_traits>

#include "dp_device.cuh"
#include "dp_internal.h"
#include "dp_launch.h"
#include "dp_single.cuh"

namespace dp {

// ============================================================================ reduce (pass A)

// (Thread and shared-memory layout, launch parameters and the single pass's shared per-tile steps:
// dp_single.cuh.)

// Single pass, gbar in registers (FUSED 2): one local element j of tile t -- Adam with gbar g on the old
// state (shared memory inside the tile's 4-aligned local interior [jlo, jhi), the current set at its ragged
// ends), the new state into the other set, the bf16 image into the staging tile at the element's global
// position in the cell.
struct SpTile {
  int64_t delta, cb, jlo, jhi;
  int cur, owner;
  const volatile int* ragged;   // the head / tail groups copied into shared memory
};
template <int MAXSEG>
__device__ __forceinline__ void sp_update1(const ReduceParams<MAXSEG>& p, const SpTile& T, const AdamK& K, float g,
                                           int64_t j, const float* s_state, uint16_t* s_stage) {
  float th, mm, vv;
  if ((j >= T.jlo && j < T.jhi) || T.ragged[j < T.jlo ? 0 : 1]) {
    const int64_t o = RA_STATE_PAD + (j - T.jlo);
    th = s_state[o];
    mm = s_state[RA_STATE_FLOATS + o];
    vv = s_state[2 * RA_STATE_FLOATS + o];
  } else {
    th = p.st_master[T.cur][T.owner][j];
    mm = p.st_m[T.cur][T.owner][j];
    vv = p.st_v[T.cur][T.owner][j];
  }
  adam1(g, th, mm, vv, K);
  p.st_master[T.cur ^ 1][T.owner][j] = th;
  p.st_m[T.cur ^ 1][T.owner][j] = mm;
  p.st_v[T.cur ^ 1][T.owner][j] = vv;
  s_stage[j - T.delta - T.cb] = bf16_rn(th);
}
// Four local elements [j, j + 4), j a multiple of 4 inside [jlo, jhi): 16-byte accesses.
template <int MAXSEG>
__device__ __forceinline__ void sp_update4(const ReduceParams<MAXSEG>& p, const SpTile& T, const AdamK& K, float g0,
                                           float g1, float g2, float g3, int64_t j, const float* s_state,
                                           uint16_t* s_stage) {
  float4 th = *reinterpret_cast<const float4*>(s_state + RA_STATE_PAD + (j - T.jlo));
  float4 mm = *reinterpret_cast<const float4*>(s_state + RA_STATE_FLOATS + RA_STATE_PAD + (j - T.jlo));
  float4 vv = *reinterpret_cast<const float4*>(s_state + 2 * RA_STATE_FLOATS + RA_STATE_PAD + (j - T.jlo));
  adam1(g0, th.x, mm.x, vv.x, K);
  adam1(g1, th.y, mm.y, vv.y, K);
  adam1(g2, th.z, mm.z, vv.z, K);
  adam1(g3, th.w, mm.w, vv.w, K);
  *reinterpret_cast<float4*>(p.st_master[T.cur ^ 1][T.owner] + j) = th;
  *reinterpret_cast<float4*>(p.st_m[T.cur ^ 1][T.owner] + j) = mm;
  *reinterpret_cast<float4*>(p.st_v[T.cur ^ 1][T.owner] + j) = vv;
  stage_bf16x4(s_stage, j - T.delta - T.cb, bf16x2_rn(th.x, th.y), bf16x2_rn(th.z, th.w));
}

// Fold input HH of a stage (8 words = 16 bf16 of this thread) into the accumulators, ring order.
//  compensated: one (H, L) pair through the whole sequence, (H, e) = TwoSum(H, x), L = L + e (first: H = x);
//  plain: each rank's micro-steps summed left to right in h (kfirst starts a rank), and at the rank's last
//  micro-step (klast) h joins the ring sum, H = ((h_{s+1} + h_{s+2}) + ...) + h_s.
template <bool COMP, int HH>
__device__ __forceinline__ void fold_input(f2_t (&H)[8], f2_t (&L)[8], f2_t (&h)[8], const uint32_t (&w)[8 * RA_NPS],
                                           bool first, bool kfirst, bool klast, bool first_rank) {
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const f2_t x = bf16x2_to_f2(w[8 * HH + u]);
    if (COMP) {
      if (first) {
        H[u] = x;
        L[u] = 0ull;
      } else {
        f2_t e;
        H[u] = f2_two_sum(H[u], x, e);
        L[u] = f2_add(L[u], e);
      }
    } else {
      h[u] = kfirst ? x : f2_add(h[u], x);
      if (klast) H[u] = first_rank ? h[u] : f2_add(H[u], h[u]);
    }
  }
}

template <int MAXSEG, bool COMP, int FUSED>
__global__ void __launch_bounds__(RA_THREADS, 1) reduce_kernel(const __grid_constant__ ReduceParams<MAXSEG> p) {
  constexpr int NST = ra_stages<FUSED>();
  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char* stages = smem;
  // single pass: the gbar tile (FUSED 1), the bf16 staging tile (global position in the cell), the tile's old
  // master, m, v (4-aligned local interior), RA_STATE_FLOATS apart
  float* s_g = reinterpret_cast<float*>(smem + NST * RA_STAGE_BYTES);
  uint16_t* s_stage = reinterpret_cast<uint16_t*>(smem + NST * RA_STAGE_BYTES + ra_gbar_bytes<FUSED>());
  float* s_state = reinterpret_cast<float*>(smem + NST * RA_STAGE_BYTES + ra_gbar_bytes<FUSED>() + TILE * 2);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + ra_bar_offset<FUSED>());
  uint64_t* empty = full + NST;
  uint64_t* sfull = empty + NST;        // single pass: the tile's state has landed (producer + bytes)
  uint64_t* sempty = sfull + 1;         // single pass: the update is done reading it (consumer warps)
  volatile int* s_abort = reinterpret_cast<volatile int*>(sfull + (FUSED ? 2 : 0));
  unsigned long long* s_count = reinterpret_cast<unsigned long long*>(sfull + (FUSED ? 2 : 0) + 1);
  __shared__ float s_inv;
  __shared__ float s_k[2];
  __shared__ int s_cur;
  __shared__ int s_ragged_buf[2];   // single pass: the current tile's head / tail state groups are in s_state
  volatile int* s_ragged = s_ragged_buf;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n = p.n, a = p.a;
  const int ntiles = p.seg.ntiles;
  const int64_t psi = p.seg.psi;
  const int64_t p8 = psi & ~int64_t(7);

  if (tid == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), RA_CWARPS);
    }
    if (FUSED) {
      mbar_init(smem_u32(sfull), 1);
      mbar_init(smem_u32(sempty), RA_CWARPS);
    }
    *s_abort = 0;
    *s_count = 0ull;
    float inv = p.inv;
    if (p.scaler.enabled) {
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
    if (FUSED) {
      // Bias corrections of the step being taken (t + 1): the same double products the finish stores.
      const volatile dp_step_state_t* vs = p.state;
      s_k[0] = (float)((double)p.lr / (1.0 - vs->b1t * p.beta1));
      s_k[1] = (float)(1.0 / sqrt(1.0 - vs->b2t * p.beta2));
      s_cur = (int)(vs->cur_set & 1u);
    }
    fence_mbar_init();
  }
  __syncthreads();

  unsigned bad = 0;
  if (warp == RA_CWARPS) {
    // ------------------------------------------------------------ producer: one thread issues every copy
    if (lane == 0) {
      RingPos<NST> rp;
      TileWalker<MAXSEG> walk;
      const int nin = n * a;
      uint32_t sit = 0;   // single pass: tiles whose state copies were issued
      for (int tile = blockIdx.x; tile < ntiles && !*s_abort; tile += gridDim.x) {
        const Tile t = walk.at(p.seg, tile);
        const int64_t A = t.start & ~int64_t(7);
        int64_t B = (t.end + 7) & ~int64_t(7);
        if (B > p8) B = p8;
        const uint32_t bytes = B > A ? (uint32_t)(B - A) * 2u : 0u;
        // Single pass: the tile's old master/m/v (4-aligned local interior, the current set) into s_state, once
        // the update of the previous tile has read it.  Issued after the tile's first NST stages, when the next
        // stage would wait for the consumers anyway.
        auto issue_state = [&]() { sp_issue_state(p, t, s_cur, sit, s_state, s_ragged, sfull, sempty, s_abort); };
        const int tile_stages = (nin + RA_NPS - 1) / RA_NPS;
        const int state_after = tile_stages < NST ? tile_stages : NST;
        int sq = 0;
        // Inputs in ring order: rank owner+1 first, its micro-steps 0..a-1, then the next rank; two per stage.
        int r = t.owner + 1 == n ? 0 : t.owner + 1, k = 0;
        for (int q = 0; q < nin && !*s_abort; q += RA_NPS) {
          if (rp.count >= (uint32_t)NST &&
              !mbar_wait_bounded(smem_u32(&empty[rp.slot]), rp.phase ^ 1u, p.timeout_ns, s_abort)) {
            if (!*s_abort) record_error(p.state, DP_ERR_TIMEOUT);
            *s_abort = 1;
            break;
          }
          const int cnt = nin - q < RA_NPS ? nin - q : RA_NPS;
          const uint32_t fb = smem_u32(&full[rp.slot]);
          mbar_arrive_expect_tx(fb, bytes * (uint32_t)cnt);
          for (int h = 0; h < cnt; ++h) {
            if (bytes)
              bulk_g2s(smem_u32(stages + rp.slot * RA_STAGE_BYTES + h * RA_IN_BYTES), p.g[r * a + k] + A, bytes, fb);
            if (++k == a) {
              k = 0;
              if (++r == n) r = 0;
            }
          }
          rp.next();
          if (FUSED && ++sq == state_after) issue_state();
        }
      }
      // Single pass: never leave with state copies in flight either.
      if (FUSED && *s_abort && sit > 0)
        (void)mbar_wait_bounded(smem_u32(sfull), (sit - 1) & 1u, p.timeout_ns, nullptr);
      // Never leave with copies in flight: wait for the newest issued phase of every slot.
      if (*s_abort) {
        const uint32_t it = rp.count;
        const uint32_t first = it > (uint32_t)NST ? it - NST : 0u;
        for (uint32_t x = first; x < it; ++x)
          (void)mbar_wait_bounded(smem_u32(&full[x % NST]), (x / NST) & 1u, p.timeout_ns, nullptr);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ consumers: 16 elements per thread
    const f2_t inv2 = f2_pack(s_inv, s_inv);
    const int nin = n * a;
    RingPos<NST> rp;
    TileWalker<MAXSEG> walk;
    bool live = true;
    uint32_t sit_c = 0;   // single pass: tiles whose state this thread has used
    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
      const Tile t = walk.at(p.seg, tile);
      const int64_t A = t.start & ~int64_t(7);
      const int64_t B = (t.end + 7) & ~int64_t(7);
      const int64_t e0 = A + RA_EPT * tid;
      const bool active = e0 < B;
      const bool tailgrp = active && (e0 + RA_EPT > p8);

      // One stage: wait for its bytes, take this thread's 16 values of each of its cnt inputs, release the slot.
      // FULL (the tile is a whole cell, every thread active, no buffer tail): plain shared loads only.
      // Otherwise inactive threads take zeros and the group holding the buffer's last partial 8 elements is
      // read from global memory (r0, k0: rank and micro-step of the stage's first input).  The shared abort
      // flag is only read inside a wait that did not succeed at once; `live` is this thread's view.
      auto take = [&](auto full_tag, int cnt, int r0, int k0, uint32_t (&w)[8 * RA_NPS]) {
        constexpr bool FULL = decltype(full_tag)::value;
        if (live && !mbar_wait_bounded(smem_u32(&full[rp.slot]), rp.phase, p.timeout_ns, s_abort)) {
          if (!*s_abort) record_error(p.state, DP_ERR_TIMEOUT);
          *s_abort = 1;
          live = false;
        }
        const unsigned char* sp = stages + rp.slot * RA_STAGE_BYTES + 2 * RA_EPT * tid;
        if constexpr (FULL) {
#pragma unroll
          for (int hh = 0; hh < RA_NPS; ++hh) {
            if (hh < cnt) {
              const uint4 v0 = *reinterpret_cast<const uint4*>(sp + hh * RA_IN_BYTES);
              const uint4 v1 = *reinterpret_cast<const uint4*>(sp + hh * RA_IN_BYTES + 16);
              w[8 * hh + 0] = v0.x; w[8 * hh + 1] = v0.y; w[8 * hh + 2] = v0.z; w[8 * hh + 3] = v0.w;
              w[8 * hh + 4] = v1.x; w[8 * hh + 5] = v1.y; w[8 * hh + 6] = v1.z; w[8 * hh + 7] = v1.w;
            }
          }
        } else {
#pragma unroll
          for (int u = 0; u < 8 * RA_NPS; ++u) w[u] = 0u;
          if (active && live) {
            int rr = r0, kk = k0;
#pragma unroll
            for (int hh = 0; hh < RA_NPS; ++hh) {
              if (hh < cnt) {
                if (!tailgrp) {
                  const uint4 v0 = *reinterpret_cast<const uint4*>(sp + hh * RA_IN_BYTES);
                  const uint4 v1 = *reinterpret_cast<const uint4*>(sp + hh * RA_IN_BYTES + 16);
                  w[8 * hh + 0] = v0.x; w[8 * hh + 1] = v0.y; w[8 * hh + 2] = v0.z; w[8 * hh + 3] = v0.w;
                  w[8 * hh + 4] = v1.x; w[8 * hh + 5] = v1.y; w[8 * hh + 6] = v1.z; w[8 * hh + 7] = v1.w;
                } else {
                  const uint16_t* src = p.g[rr * a + kk];
#pragma unroll
                  for (int u = 0; u < RA_EPT; ++u) {
                    const uint32_t b = (e0 + u < psi) ? (uint32_t)src[e0 + u] : 0u;
                    w[8 * hh + (u >> 1)] |= (u & 1) ? (b << 16) : b;
                  }
                }
              }
              if (++kk == a) {
                kk = 0;
                if (++rr == n) rr = 0;
              }
            }
          }
        }
        // The slot is refilled by the async proxy (bulk copy): order this thread's generic-proxy reads of
        // it before that write, then release the slot.
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty[rp.slot]));
        rp.next();
      };

      // Inputs in ring order: rank owner+1 with its micro-steps 0..a-1, then owner+2, ..., owner.  Whole
      // stages first (two inputs each, no per-input guards), then a last single input when n*a is odd.
      f2_t H[8], L[8], h[8];
      auto run = [&](auto full_tag) {
        int r = t.owner + 1 == n ? 0 : t.owner + 1, k = 0;
        bool first_rank = true;
        auto advance = [&]() {
          if (++k == a) {
            k = 0;
            first_rank = false;
            if (++r == n) r = 0;
          }
        };
        int q = 0;
        for (; q + RA_NPS <= nin; q += RA_NPS) {
          uint32_t w[8 * RA_NPS];
          take(full_tag, RA_NPS, r, k, w);
          fold_input<COMP, 0>(H, L, h, w, q == 0, k == 0, k == a - 1, first_rank);
          advance();
          fold_input<COMP, 1>(H, L, h, w, false, k == 0, k == a - 1, first_rank);
          advance();
        }
        if (q < nin) {
          uint32_t w[8 * RA_NPS];
          take(full_tag, 1, r, k, w);
          fold_input<COMP, 0>(H, L, h, w, q == 0, k == 0, k == a - 1, first_rank);
        }
      };
      static_assert(RA_NPS == 2, "the stage loop folds two inputs");
      // A whole cell is TILE-aligned, so every thread of it is active; t.end <= p8 keeps the tail group out.
      if (t.end - t.start == TILE && t.end <= p8) run(std::true_type{});
      else run(std::false_type{});

      // gbar = fl(p * inv) for the 16 elements; count the non-finite ones of this tile.
      float o[RA_EPT];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const f2_t pp = COMP ? f2_add(H[u], L[u]) : H[u];
        f2_unpack(f2_mul(pp, inv2), o[2 * u], o[2 * u + 1]);
      }
      const bool whole = active && e0 >= t.start && e0 + RA_EPT <= t.end;
      if (active) {
#pragma unroll
        for (int u = 0; u < RA_EPT; ++u)
          if ((whole || (e0 + u >= t.start && e0 + u < t.end)) && nonfinite(o[u])) ++bad;
      }
      if constexpr (FUSED != 0) {
        const int64_t cb = (t.start / TILE) * TILE;
        if constexpr (FUSED == 1) {
          // Hand the tile's gbar to its update through shared memory (indexed by global position).
          named_bar_sync(1, RA_CTHREADS);    // the previous tile's update is done with s_g and s_stage
          if (tid == 0) bulk_wait_read<0>(); // and its replica stores have read s_stage
          if (active) {
            float4* gp = reinterpret_cast<float4*>(s_g + (e0 - cb));
#pragma unroll
            for (int u = 0; u < RA_EPT; u += 4) gp[u / 4] = make_float4(o[u], o[u + 1], o[u + 2], o[u + 3]);
          }
          named_bar_sync(1, RA_CTHREADS);
        } else {
          if (tid == 0) bulk_wait_read<0>(); // the previous tile's replica stores have read s_stage
          named_bar_sync(1, RA_CTHREADS);
        }
        AdamK K;
        K.b1 = p.b1f; K.b2 = p.b2f; K.omb1 = p.omb1; K.omb2 = p.omb2; K.eps = p.eps;
        K.step = s_k[0];
        K.rsbc2 = s_k[1];
        // The tile's old state, bulk-copied by the producer while the gradients streamed.
        if (live && !mbar_wait_bounded(smem_u32(sfull), sit_c & 1u, p.timeout_ns, s_abort)) {
          if (!*s_abort) record_error(p.state, DP_ERR_TIMEOUT);
          *s_abort = 1;
          live = false;
        }
        if constexpr (FUSED == 1) {
          fused_update(p, t, K, s_cur, s_g, s_stage, s_state, s_ragged, tid);
        } else {
          // Every thread updates the elements whose gbar it holds: with every shard offset a multiple of 4 (the
          // launcher's condition for this variant) a thread's 16 elements are four aligned 4-groups in local
          // space too; a group at a segment edge is updated element by element.
          SpTile T;
          T.delta = t.loff - t.goff;
          T.cb = cb;
          T.jlo = (t.start + T.delta + 3) & ~int64_t(3);
          T.jhi = (t.end + T.delta) & ~int64_t(3);
          T.cur = s_cur;
          T.owner = t.owner;
          T.ragged = s_ragged;
          const int64_t Lt = e0 + T.delta;
          if (whole && (Lt & 3) == 0) {
#pragma unroll
            for (int u = 0; u < RA_EPT; u += 4)
              sp_update4(p, T, K, o[u], o[u + 1], o[u + 2], o[u + 3], Lt + u, s_state, s_stage);
          } else if (active) {
#pragma unroll
            for (int u = 0; u < RA_EPT; ++u)
              if (e0 + u >= t.start && e0 + u < t.end) sp_update1(p, T, K, o[u], Lt + u, s_state, s_stage);
          }
        }
        // Order this thread's reads of s_state (and writes of s_stage) before the async proxy's next use of
        // them, then hand s_state back to the producer.
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(sempty));
        ++sit_c;
        named_bar_sync(1, RA_CTHREADS);
        // All-gather: the staged bf16 tile into every replica.
        sp_gather(p, t, cb, s_stage, n, tid);
        continue;
      }
      // Store into the owner's shard at local index.  A thread's 16 values sit at local [Lt, Lt + 16).
      float* dst = p.gbar[t.owner] + (t.loff - t.goff + e0);
      const int mis = (int)((t.loff - t.goff + e0) & 3);   // the same for every thread of the tile
      const bool warp_whole = __all_sync(0xFFFFFFFFu, whole);
      if (whole && mis == 0) {
#pragma unroll
        for (int u = 0; u < RA_EPT; u += 4)
          *reinterpret_cast<float4*>(dst + u) = make_float4(o[u], o[u + 1], o[u + 2], o[u + 3]);
      } else if (warp_whole) {
        // Misaligned shard: shift by d = 4 - mis values so every lane stores one 16-byte-aligned chunk
        // [Lt + d, Lt + d + 16), borrowing d values from the next lane; lane 0 also writes its first d
        // values, lane 31 (whose next lane is in another warp) writes its own last 16 - d.
        const int d = 4 - mis;
        float nb[3];
#pragma unroll
        for (int u = 0; u < 3; ++u) nb[u] = __shfl_down_sync(0xFFFFFFFFu, o[u], 1);
        if (lane == 0) {
#pragma unroll
          for (int u = 0; u < 3; ++u)
            if (u < d) dst[u] = o[u];
        }
        if (lane != 31) {
          float c[RA_EPT];
#pragma unroll
          for (int u = 0; u < RA_EPT; ++u) {
            // c[u] = o[u + d] when that is one of this lane's values, else nb[u + d - 16]
            float own = o[RA_EPT - 1];
#pragma unroll
            for (int q = 1; q <= 3; ++q)
              if (d == q && u + q < RA_EPT) own = o[u + q];
            float bor = nb[0];
#pragma unroll
            for (int q = 1; q <= 3; ++q)
              if (d == q && u + q >= RA_EPT) bor = nb[u + q - RA_EPT];
            c[u] = (u + d < RA_EPT) ? own : bor;
          }
#pragma unroll
          for (int u = 0; u < RA_EPT; u += 4)
            *reinterpret_cast<float4*>(dst + d + u) = make_float4(c[u], c[u + 1], c[u + 2], c[u + 3]);
        } else {
#pragma unroll
          for (int u = 1; u < RA_EPT; ++u)
            if (u >= d) dst[u] = o[u];
        }
      } else if (active) {
#pragma unroll
        for (int u = 0; u < RA_EPT; ++u)
          if (e0 + u >= t.start && e0 + u < t.end) dst[u] = o[u];
      }
    }
  }

  // ------------------------------------------------------------ CTA total, then the grid's
  unsigned long long c = bad;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) c += __shfl_xor_sync(0xFFFFFFFFu, c, off);
  __syncthreads();
  if (lane == 0 && c) atomicAdd(s_count, c);
  __syncthreads();
  if (FUSED && tid == 0) bulk_wait_all();   // the last tile's replica stores
  if (tid == 0)
    finish_reduction(p.state, *s_count, (*s_count != 0ull) || *s_abort, p.advance, p.beta1, p.beta2, &p.scaler,
                     FUSED ? 1 : 0, p.merge);
}

// ============================================================================ update (pass B)

constexpr int UB_THREADS = 512;
constexpr int UB_GROUPS = (TILE / 4 + UB_THREADS - 1) / UB_THREADS;  // 4-element groups per thread per tile
static_assert(UB_GROUPS * 4 * UB_THREADS >= TILE + 4, "a tile's 4-groups (one extra when misaligned) fit");

template <int MAXSEG>
struct UpdateParams {
  uint16_t* rep[DP_MAX_N];
  float* master[DP_MAX_N];
  float* m[DP_MAX_N];
  float* v[DP_MAX_N];
  const float* gbar[DP_MAX_N];
  const dp_step_state_t* state;
  float lr, beta1, beta2, eps, omb1, omb2;
  int32_t n;
  SegTable<MAXSEG> seg;
};

__device__ __forceinline__ bool update_prologue(const dp_step_state_t* st, float lr, AdamK& K, float* s_k) {
  const volatile dp_step_state_t* vs = st;
  if (vs->found_inf || vs->t == 0) return false;   // skipped step, or no reduction ran
  if (threadIdx.x == 0) {
    const double bc1 = 1.0 - vs->b1t, bc2 = 1.0 - vs->b2t;
    s_k[0] = (float)((double)lr / bc1);
    s_k[1] = (float)(1.0 / sqrt(bc2));
  }
  __syncthreads();
  K.step = s_k[0];
  K.rsbc2 = s_k[1];
  return true;
}


// Stages 1-3: shard arrays in local index space.  REPL: also all-gather.
template <int MAXSEG, bool REPL>
__global__ void __launch_bounds__(UB_THREADS) update_kernel(const __grid_constant__ UpdateParams<MAXSEG> p) {
  __shared__ __align__(128) uint16_t sbuf[REPL ? 2 : 1][REPL ? TILE : 8];
  __shared__ float s_k[2];
  AdamK K;
  K.b1 = p.beta1; K.b2 = p.beta2; K.omb1 = p.omb1; K.omb2 = p.omb2; K.eps = p.eps;
  if (!update_prologue(p.state, p.lr, K, s_k)) return;
  const int tid = threadIdx.x;
  const int ntiles = p.seg.ntiles;
  int it = 0;
  for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++it) {
    const Tile t = tile_at(p.seg, tile);
    const int64_t delta = t.loff - t.goff;
    const int64_t js = t.start + delta, je = t.end + delta;
    const int64_t jlo = (js + 3) & ~int64_t(3), jhi = je & ~int64_t(3);
    const int ngr = jhi > jlo ? (int)((jhi - jlo) >> 2) : 0;
    const int64_t cb = (t.start / TILE) * TILE;
    float* __restrict__ M = p.master[t.owner];
    float* __restrict__ Mm = p.m[t.owner];
    float* __restrict__ Vv = p.v[t.owner];
    const float* __restrict__ G = p.gbar[t.owner];
    uint16_t* sb = sbuf[REPL ? (it & 1) : 0];
    if (REPL) {
      if (tid == 0) bulk_wait_read<1>();  // the bulk stores of two tiles ago have read this buffer
      __syncthreads();
    }
    float4 g4[UB_GROUPS], t4[UB_GROUPS], m4[UB_GROUPS], v4[UB_GROUPS];
#pragma unroll
    for (int u = 0; u < UB_GROUPS; ++u) {
      const int gq = tid + u * UB_THREADS;
      if (gq < ngr) {
        const int64_t jj = jlo + 4 * (int64_t)gq;
        g4[u] = __ldcs(reinterpret_cast<const float4*>(G + jj));
        t4[u] = *reinterpret_cast<const float4*>(M + jj);
        m4[u] = *reinterpret_cast<const float4*>(Mm + jj);
        v4[u] = *reinterpret_cast<const float4*>(Vv + jj);
      }
    }
#pragma unroll
    for (int u = 0; u < UB_GROUPS; ++u) {
      const int gq = tid + u * UB_THREADS;
      if (gq < ngr) {
        const int64_t jj = jlo + 4 * (int64_t)gq;
        adam1(g4[u].x, t4[u].x, m4[u].x, v4[u].x, K);
        adam1(g4[u].y, t4[u].y, m4[u].y, v4[u].y, K);
        adam1(g4[u].z, t4[u].z, m4[u].z, v4[u].z, K);
        adam1(g4[u].w, t4[u].w, m4[u].w, v4[u].w, K);
        *reinterpret_cast<float4*>(M + jj) = t4[u];
        *reinterpret_cast<float4*>(Mm + jj) = m4[u];
        *reinterpret_cast<float4*>(Vv + jj) = v4[u];
        if (REPL) stage_bf16x4(sb, jj - delta - cb, bf16x2_rn(t4[u].x, t4[u].y), bf16x2_rn(t4[u].z, t4[u].w));
      }
    }
    // Ragged ends of the tile in local space (at most 3 elements each): scalar.
    {
      int64_t jx = -1;
      if (tid < 4) {
        jx = js + tid;
        if (jx >= (jlo < je ? jlo : je)) jx = -1;
      } else if (tid < 8) {
        jx = (jhi > jlo ? jhi : jlo) + (tid - 4);
        if (jx >= je) jx = -1;
      }
      if (jx >= 0) {
        float th = M[jx], mm = Mm[jx], vv = Vv[jx];
        adam1(G[jx], th, mm, vv, K);
        M[jx] = th;
        Mm[jx] = mm;
        Vv[jx] = vv;
        if (REPL) sb[jx - delta - cb] = bf16_rn(th);
      }
    }
    if (REPL) {
      fence_proxy_async_smem();
      __syncthreads();
      const int64_t ilo = (t.start + 7) & ~int64_t(7), ihi = t.end & ~int64_t(7);
      if (tid == 0) {
        if (ihi > ilo) {
          const uint32_t src = smem_u32(sb + (ilo - cb));
          const uint32_t bytes = (uint32_t)(ihi - ilo) * 2u;
          for (int r = 0; r < p.n; ++r) bulk_s2g(p.rep[r] + ilo, src, bytes);
        }
        bulk_commit();
      }
      // Global-space ragged ends (fewer than 8 elements each) with plain stores.
      if (tid < 16) {
        int64_t ix = -1;
        if (tid < 8) {
          ix = t.start + tid;
          if (ix >= (ilo < t.end ? ilo : t.end)) ix = -1;
        } else {
          ix = (ihi > ilo ? ihi : ilo) + (tid - 8);
          if (ix >= t.end) ix = -1;
        }
        if (ix >= 0) {
          const uint16_t b = sb[ix - cb];
          for (int r = 0; r < p.n; ++r) p.rep[r][ix] = b;
        }
      }
    }
  }
  if (REPL && tid == 0) bulk_wait_all();
}

// Stage 0 (plain data parallelism): every rank updates its own full-length state with the owner's gbar, and
// writes its own replica.  The work items of a tile are (rank, 4-element group) pairs of its 4-aligned global
// interior, rank-major so that a warp's items are consecutive groups of one rank: each item reads the group's
// master, m, v as 16-byte vectors at global index, writes them back and stores its four bf16 as one 8-byte
// word.  The n items of a group read the same gbar vector (the tile's gbar, 30 KB, is served by L1/L2 after
// the first).  UB_GROUPS items per thread have their loads issued before any arithmetic.  The <= 3 elements at
// each end of the tile are updated one by one.
template <int MAXSEG, bool REPL>
__global__ void __launch_bounds__(UB_THREADS) update_dp_kernel(const __grid_constant__ UpdateParams<MAXSEG> p) {
  __shared__ float s_k[2];
  AdamK K;
  K.b1 = p.beta1; K.b2 = p.beta2; K.omb1 = p.omb1; K.omb2 = p.omb2; K.eps = p.eps;
  if (!update_prologue(p.state, p.lr, K, s_k)) return;
  const int tid = threadIdx.x, n = p.n;
  const int ntiles = p.seg.ntiles;
  for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    const Tile t = tile_at(p.seg, tile);
    const float* __restrict__ G = p.gbar[t.owner];
    const int64_t delta = t.loff - t.goff;            // gbar's local index = global index + delta
    const bool galign = (delta & 3) == 0;
    const int64_t elo = (t.start + 3) & ~int64_t(3), ehi = t.end & ~int64_t(3);
    const int ngr = ehi > elo ? (int)((ehi - elo) >> 2) : 0;
    const int items = ngr * n;
    for (int base = 0; base < items; base += UB_GROUPS * UB_THREADS) {
      float4 g4[UB_GROUPS], t4[UB_GROUPS], m4[UB_GROUPS], v4[UB_GROUPS];
      int rr[UB_GROUPS];
      int64_t ee[UB_GROUPS];
#pragma unroll
      for (int u = 0; u < UB_GROUPS; ++u) {
        const int w = base + tid + u * UB_THREADS;
        rr[u] = -1;
        if (w < items) {
          const int r = w / ngr;
          const int64_t e = elo + 4 * (int64_t)(w - r * ngr);
          rr[u] = r;
          ee[u] = e;
          const float* gs = G + (e + delta);
          g4[u] = galign ? *reinterpret_cast<const float4*>(gs) : make_float4(gs[0], gs[1], gs[2], gs[3]);
          t4[u] = __ldcs(reinterpret_cast<const float4*>(p.master[r] + e));
          m4[u] = __ldcs(reinterpret_cast<const float4*>(p.m[r] + e));
          v4[u] = __ldcs(reinterpret_cast<const float4*>(p.v[r] + e));
        }
      }
#pragma unroll
      for (int u = 0; u < UB_GROUPS; ++u) {
        if (rr[u] >= 0) {
          const int r = rr[u];
          const int64_t e = ee[u];
          adam1(g4[u].x, t4[u].x, m4[u].x, v4[u].x, K);
          adam1(g4[u].y, t4[u].y, m4[u].y, v4[u].y, K);
          adam1(g4[u].z, t4[u].z, m4[u].z, v4[u].z, K);
          adam1(g4[u].w, t4[u].w, m4[u].w, v4[u].w, K);
          __stcs(reinterpret_cast<float4*>(p.master[r] + e), t4[u]);
          __stcs(reinterpret_cast<float4*>(p.m[r] + e), m4[u]);
          __stcs(reinterpret_cast<float4*>(p.v[r] + e), v4[u]);
          if (REPL)
            __stcs(reinterpret_cast<uint2*>(p.rep[r] + e),
                   make_uint2(bf16x2_rn(t4[u].x, t4[u].y), bf16x2_rn(t4[u].z, t4[u].w)));
        }
      }
    }
    // Ragged ends (at most 3 elements each) of every rank: thread 8r + k, k < 4 the head, k >= 4 the tail.
    if (tid < 8 * n) {
      const int r = tid >> 3, k = tid & 7;
      int64_t e = -1;
      if (k < 4) {
        e = t.start + k;
        if (e >= (elo < t.end ? elo : t.end)) e = -1;
      } else {
        e = (ehi > elo ? ehi : elo) + (k - 4);
        if (e >= t.end) e = -1;
      }
      if (e >= 0) {
        float th = p.master[r][e], mm = p.m[r][e], vv = p.v[r][e];
        adam1(G[e + delta], th, mm, vv, K);
        p.master[r][e] = th;
        p.m[r][e] = mm;
        p.v[r][e] = vv;
        if (REPL) p.rep[r][e] = bf16_rn(th);
      }
    }
  }
}

// ============================================================================ staged kernels

struct AccParams {
  float* acc[DP_MAX_N];
  const uint16_t* g[DP_MAX_N];
  int64_t psi;
  int32_t n, first;
};

template <bool COMP>
__global__ void __launch_bounds__(256) accumulate_kernel(const __grid_constant__ AccParams p) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < p.psi; e += stride) {
    for (int r = 0; r < p.n; ++r) {
      const float x = bf16_to_f32(p.g[r][e]);
      if (COMP) {
        float2* a2 = reinterpret_cast<float2*>(p.acc[r]) + e;
        if (p.first) {
          *a2 = make_float2(x, 0.0f);
        } else {
          float2 hl = *a2;
          float err;
          hl.x = two_sum(hl.x, x, err);
          hl.y = __fadd_rn(hl.y, err);
          *a2 = hl;
        }
      } else {
        float* a1 = p.acc[r] + e;
        *a1 = p.first ? x : __fadd_rn(*a1, x);
      }
    }
  }
}

template <int MAXSEG>
struct RsParams {
  const float* acc[DP_MAX_N];
  float* gbar[DP_MAX_N];
  dp_step_state_t* state;
  float inv;
  int32_t n, merge;
  SegTable<MAXSEG> seg;
};

template <int MAXSEG, bool COMP>
__global__ void __launch_bounds__(256) rs_avg_kernel(const __grid_constant__ RsParams<MAXSEG> p) {
  __shared__ unsigned long long s_count;
  if (threadIdx.x == 0) s_count = 0ull;
  __syncthreads();
  unsigned bad = 0;
  const int n = p.n;
  for (int tile = blockIdx.x; tile < p.seg.ntiles; tile += gridDim.x) {
    const Tile t = tile_at(p.seg, tile);
    float* dst = p.gbar[t.owner];
    for (int64_t e = t.start + threadIdx.x; e < t.end; e += blockDim.x) {
      int r = t.owner + 1 == n ? 0 : t.owner + 1;
      float H = 0.0f, L = 0.0f;
      for (int j = 0; j < n; ++j) {
        if (COMP) {
          const float2 hl = reinterpret_cast<const float2*>(p.acc[r])[e];
          if (j == 0) {
            H = hl.x;
            L = hl.y;
          } else {
            float err;
            H = two_sum(H, hl.x, err);
            L = __fadd_rn(L, err);
            L = __fadd_rn(L, hl.y);
          }
        } else {
          const float h = p.acc[r][e];
          H = (j == 0) ? h : __fadd_rn(H, h);
        }
        if (++r == n) r = 0;
      }
      const float pp = COMP ? __fadd_rn(H, L) : H;
      const float g = __fmul_rn(pp, p.inv);
      dst[t.loff + (e - t.goff)] = g;
      if (nonfinite(g)) ++bad;
    }
  }
  unsigned long long c = bad;
  for (int off = 16; off > 0; off >>= 1) c += __shfl_xor_sync(0xFFFFFFFFu, c, off);
  if ((threadIdx.x & 31) == 0 && c) atomicAdd(&s_count, c);
  __syncthreads();
  if (threadIdx.x == 0) finish_reduction(p.state, s_count, s_count != 0ull, 0, 1.0, 1.0, nullptr, 0, p.merge);
}

template <int MAXSEG>
struct AgParams {
  uint16_t* rep[DP_MAX_N];
  const float* master[DP_MAX_N];
  const dp_step_state_t* state;
  int32_t n, stage;
  SegTable<MAXSEG> seg;
};

template <int MAXSEG>
__global__ void __launch_bounds__(256) allgather_kernel(const __grid_constant__ AgParams<MAXSEG> p) {
  const volatile dp_step_state_t* vs = p.state;
  if (vs->found_inf) return;
  for (int tile = blockIdx.x; tile < p.seg.ntiles; tile += gridDim.x) {
    const Tile t = tile_at(p.seg, tile);
    for (int64_t e = t.start + threadIdx.x; e < t.end; e += blockDim.x) {
      if (p.stage == 0) {
        for (int r = 0; r < p.n; ++r) p.rep[r][e] = bf16_rn(p.master[r][e]);
      } else {
        const uint16_t b = bf16_rn(p.master[t.owner][t.loff + (e - t.goff)]);
        for (int r = 0; r < p.n; ++r) p.rep[r][e] = b;
      }
    }
  }
}

__global__ void advance_kernel(dp_step_state_t* st, double b1, double b2) {
  if (!st->found_inf) {
    st->t += 1;
    st->b1t *= b1;
    st->b2t *= b2;
  }
}

// The commit of a step whose reduction deferred it: found_inf now holds the decision of every slice (a
// recorded device error also skips the step).
__global__ void commit_kernel(dp_step_state_t* st, double b1, double b2, ScalerK scaler, int flip_set) {
  const int err = st->error;
  const int found = (st->found_inf != 0 || err != 0) ? 1 : 0;
  st->found_inf = found;
  commit_state(st, found, err, b1, b2, &scaler, flip_set);
}

__global__ void state_init_kernel(dp_step_state_t* st) {
  st->t = 0;
  st->found_inf = 0;
  st->error = 0;
  st->good_steps = 0;
  st->loss_scale = 0.0f;
  st->cur_set = 0u;
  st->nonfinite = 0ull;
  st->b1t = 1.0;
  st->b2t = 1.0;
  st->work_count = 0ull;
  st->work_found = 0u;
  st->work_ticket = 0u;
}

__global__ void scaler_init_kernel(dp_step_state_t* st, float scale) {
  st->loss_scale = scale;
  st->good_steps = 0;
}

// One block waits on a barrier that expects two arrivals but receives one.
__global__ void selftest_wait_kernel(dp_step_state_t* st, uint64_t timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 2);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    mbar_arrive(smem_u32(&bar));
    if (!mbar_wait_bounded(smem_u32(&bar), 0u, timeout_ns, nullptr)) record_error(st, DP_ERR_TIMEOUT);
  }
}

// ============================================================================ launchers




template <int MAXSEG, bool COMP, int FUSED>
static cudaError_t launch_reduce_t(const Plan& P, const uint16_t* const* g, int a, float* const* gbar,
                                   const StepScalars& s, int advance, dp_step_state_t* st, const FusedArgs* fa,
                                   cudaStream_t stream) {
  ReduceParams<MAXSEG> prm;
  fill_reduce_params(prm, P, g, a, gbar, s, advance, st, fa);
  auto kern = reduce_kernel<MAXSEG, COMP, FUSED>;
  constexpr int smem = ra_smem<FUSED>();
  // The opt-in shared-memory size is set once per device (not inside a stream capture on later calls).
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  // Every CTA takes part in the grid-wide finish, so at least one CTA runs even with no tiles.
  int grid = sm_count();
  if (P.ntiles < grid) grid = P.ntiles > 0 ? P.ntiles : 1;
  kern<<<grid, RA_THREADS, smem, stream>>>(prm);
  return cudaGetLastError();
}

cudaError_t launch_reduce(const Plan& P0, const uint16_t* const* g, int a, float* const* gbar,
                          const StepScalars& s0, int advance0, dp_step_state_t* st, cudaStream_t stream,
                          uint64_t* launches) {
  return for_each_chunk(P0, s0, [&](const Plan& P, const StepScalars& s, bool last) {
    ++*launches;
    const int advance = (advance0 && last) ? 1 : 0;
    const bool comp = s.mode == DP_SUM_COMPENSATED;
    if (P.nseg <= SMALL_SEG)
      return comp ? launch_reduce_t<SMALL_SEG, true, 0>(P, g, a, gbar, s, advance, st, nullptr, stream)
                  : launch_reduce_t<SMALL_SEG, false, 0>(P, g, a, gbar, s, advance, st, nullptr, stream);
    return comp ? launch_reduce_t<BIG_SEG, true, 0>(P, g, a, gbar, s, advance, st, nullptr, stream)
                : launch_reduce_t<BIG_SEG, false, 0>(P, g, a, gbar, s, advance, st, nullptr, stream);
  });
}

// After a single-pass step: if it was skipped, rewrite the replicas as bf16 of the current (unchanged) master.
template <int MAXSEG>
struct RepairParams {
  uint16_t* rep[DP_MAX_N];
  const float* master[2][DP_MAX_N];
  const dp_step_state_t* state;
  int32_t n;
  SegTable<MAXSEG> seg;
};

template <int MAXSEG>
__global__ void __launch_bounds__(256) repair_kernel(const __grid_constant__ RepairParams<MAXSEG> p) {
  const volatile dp_step_state_t* vs = p.state;
  if (!vs->found_inf) return;
  const int cur = (int)(vs->cur_set & 1u);
  for (int tile = blockIdx.x; tile < p.seg.ntiles; tile += gridDim.x) {
    const Tile t = tile_at(p.seg, tile);
    const float* M = p.master[cur][t.owner];
    for (int64_t e = t.start + threadIdx.x; e < t.end; e += blockDim.x) {
      const uint16_t b = bf16_rn(M[t.loff + (e - t.goff)]);
      for (int r = 0; r < p.n; ++r) p.rep[r][e] = b;
    }
  }
}

template <int MAXSEG>
static cudaError_t launch_repair_t(const Plan& P, uint16_t* const* rep, float* const* master2,
                                   const dp_step_state_t* st, cudaStream_t stream) {
  RepairParams<MAXSEG> rp;
  for (int r = 0; r < P.n; ++r) {
    rp.rep[r] = rep[r];
    rp.master[0][r] = master2[r];
    rp.master[1][r] = master2[P.n + r];
  }
  rp.state = st;
  rp.n = P.n;
  fill_seg(rp.seg, P);
  auto k = repair_kernel<MAXSEG>;
  k<<<occupancy_grid(k, 256, 0, P.ntiles > 0 ? P.ntiles : 1), 256, 0, stream>>>(rp);
  return cudaGetLastError();
}

template <int MAXSEG>
static cudaError_t launch_single_t(const Plan& P, const uint16_t* const* g, int a, const StepScalars& s,
                                   dp_step_state_t* st, const FusedArgs& fa, cudaStream_t stream) {
  // gbar stays in registers when every shard offset keeps 4-groups aligned and a tile has enough inputs for the
  // fourth stage to pay; otherwise the shared gbar tile regroups it.
  bool realign = P.n * a >= 16;
  for (int k = 0; k < P.nseg; ++k)
    if (((P.e[k].loff - P.e[k].goff) & 3) != 0) realign = false;
  const bool comp = s.mode == DP_SUM_COMPENSATED;
  const int adv = s.defer ? 0 : 1;
  cudaError_t e = realign ? (comp ? launch_reduce_t<MAXSEG, true, 2>(P, g, a, nullptr, s, adv, st, &fa, stream)
                                  : launch_reduce_t<MAXSEG, false, 2>(P, g, a, nullptr, s, adv, st, &fa, stream))
                          : (comp ? launch_reduce_t<MAXSEG, true, 1>(P, g, a, nullptr, s, adv, st, &fa, stream)
                                  : launch_reduce_t<MAXSEG, false, 1>(P, g, a, nullptr, s, adv, st, &fa, stream));
  return e;
}

cudaError_t launch_single_pass(const Plan& P0, const uint16_t* const* g, int a, uint16_t* const* rep,
                               float* const* master2, float* const* m2, float* const* v2, const StepScalars& s0,
                               dp_step_state_t* st, cudaStream_t stream, uint64_t* launches) {
  const FusedArgs fa{master2, m2, v2, rep};
  cudaError_t e = for_each_chunk(P0, s0, [&](const Plan& P, const StepScalars& s, bool) {
    ++*launches;
    if (s.order == DP_ORDER_TREE) return launch_tree_single(P, g, a, s, st, fa, stream);
    if (P.nseg <= SMALL_SEG) return launch_single_t<SMALL_SEG>(P, g, a, s, st, fa, stream);
    return launch_single_t<BIG_SEG>(P, g, a, s, st, fa, stream);
  });
  if (e != cudaSuccess || s0.defer) return e;   // deferred: the commit call launches the repair
  return launch_repair(P0, rep, master2, st, stream, launches);
}

template <int MAXSEG>
static cudaError_t launch_update_t(const Plan& P, uint16_t* const* rep, float* const* master, float* const* m,
                                   float* const* v, const float* const* gbar, const StepScalars& s,
                                   const dp_step_state_t* st, cudaStream_t stream) {
  UpdateParams<MAXSEG> prm;
  for (int r = 0; r < P.n; ++r) {
    prm.rep[r] = rep ? rep[r] : nullptr;
    prm.master[r] = master[r];
    prm.m[r] = m[r];
    prm.v[r] = v[r];
    prm.gbar[r] = gbar[r];
  }
  prm.state = st;
  prm.lr = s.lr;
  prm.beta1 = s.beta1;
  prm.beta2 = s.beta2;
  prm.eps = s.eps;
  prm.omb1 = s.omb1;
  prm.omb2 = s.omb2;
  prm.n = P.n;
  fill_seg(prm.seg, P);
  const int nt = P.ntiles > 0 ? P.ntiles : 1;
  if (P.stage == 0) {
    if (rep) {
      auto k = update_dp_kernel<MAXSEG, true>;
      k<<<occupancy_grid(k, UB_THREADS, 0, nt), UB_THREADS, 0, stream>>>(prm);
    } else {
      auto k = update_dp_kernel<MAXSEG, false>;
      k<<<occupancy_grid(k, UB_THREADS, 0, nt), UB_THREADS, 0, stream>>>(prm);
    }
  } else {
    if (rep) {
      auto k = update_kernel<MAXSEG, true>;
      k<<<occupancy_grid(k, UB_THREADS, 0, nt), UB_THREADS, 0, stream>>>(prm);
    } else {
      auto k = update_kernel<MAXSEG, false>;
      k<<<occupancy_grid(k, UB_THREADS, 0, nt), UB_THREADS, 0, stream>>>(prm);
    }
  }
  return cudaGetLastError();
}

cudaError_t launch_update(const Plan& P0, uint16_t* const* rep, float* const* master, float* const* m,
                          float* const* v, const float* const* gbar, const StepScalars& s0,
                          const dp_step_state_t* st, cudaStream_t stream, uint64_t* launches) {
  return for_each_chunk(P0, s0, [&](const Plan& P, const StepScalars& s, bool) {
    ++*launches;
    if (P.nseg <= SMALL_SEG) return launch_update_t<SMALL_SEG>(P, rep, master, m, v, gbar, s, st, stream);
    return launch_update_t<BIG_SEG>(P, rep, master, m, v, gbar, s, st, stream);
  });
}

cudaError_t launch_accumulate(float* const* acc, const uint16_t* const* g, int64_t psi, int n, int first, int mode,
                              cudaStream_t stream, uint64_t* launches) {
  ++*launches;
  AccParams prm;
  for (int r = 0; r < n; ++r) {
    prm.acc[r] = acc[r];
    prm.g[r] = g[r];
  }
  prm.psi = psi;
  prm.n = n;
  prm.first = first ? 1 : 0;
  long long blocks = (psi + 255) / 256;
  const long long cap = (long long)sm_count() * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  if (mode == DP_SUM_COMPENSATED)
    accumulate_kernel<true><<<(int)blocks, 256, 0, stream>>>(prm);
  else
    accumulate_kernel<false><<<(int)blocks, 256, 0, stream>>>(prm);
  return cudaGetLastError();
}

template <int MAXSEG>
static cudaError_t launch_rs_t(const Plan& P, const float* const* acc, float* const* gbar, const StepScalars& s,
                               dp_step_state_t* st, cudaStream_t stream) {
  RsParams<MAXSEG> prm;
  for (int r = 0; r < P.n; ++r) {
    prm.acc[r] = acc[r];
    prm.gbar[r] = gbar[r];
  }
  prm.state = st;
  prm.inv = s.inv;
  prm.n = P.n;
  prm.merge = s.merge;
  fill_seg(prm.seg, P);
  const int nt = P.ntiles > 0 ? P.ntiles : 1;
  if (s.mode == DP_SUM_COMPENSATED) {
    auto k = rs_avg_kernel<MAXSEG, true>;
    k<<<occupancy_grid(k, 256, 0, nt), 256, 0, stream>>>(prm);
  } else {
    auto k = rs_avg_kernel<MAXSEG, false>;
    k<<<occupancy_grid(k, 256, 0, nt), 256, 0, stream>>>(prm);
  }
  return cudaGetLastError();
}

cudaError_t launch_rs_avg(const Plan& P0, const float* const* acc, float* const* gbar, const StepScalars& s0,
                          dp_step_state_t* st, cudaStream_t stream, uint64_t* launches) {
  return for_each_chunk(P0, s0, [&](const Plan& P, const StepScalars& s, bool) {
    ++*launches;
    if (P.nseg <= SMALL_SEG) return launch_rs_t<SMALL_SEG>(P, acc, gbar, s, st, stream);
    return launch_rs_t<BIG_SEG>(P, acc, gbar, s, st, stream);
  });
}

cudaError_t launch_advance(dp_step_state_t* st, double b1, double b2, cudaStream_t stream, uint64_t* launches) {
  ++*launches;
  advance_kernel<<<1, 1, 0, stream>>>(st, b1, b2);
  return cudaGetLastError();
}

template <int MAXSEG>
static cudaError_t launch_ag_t(const Plan& P, uint16_t* const* rep, const float* const* master,
                               const dp_step_state_t* st, cudaStream_t stream) {
  AgParams<MAXSEG> prm;
  for (int r = 0; r < P.n; ++r) {
    prm.rep[r] = rep[r];
    prm.master[r] = master[r];
  }
  prm.state = st;
  prm.n = P.n;
  prm.stage = P.stage;
  fill_seg(prm.seg, P);
  auto k = allgather_kernel<MAXSEG>;
  k<<<occupancy_grid(k, 256, 0, P.ntiles > 0 ? P.ntiles : 1), 256, 0, stream>>>(prm);
  return cudaGetLastError();
}

cudaError_t launch_allgather(const Plan& P0, uint16_t* const* rep, const float* const* master,
                             const dp_step_state_t* st, cudaStream_t stream, uint64_t* launches) {
  StepScalars s0{};
  return for_each_chunk(P0, s0, [&](const Plan& P, const StepScalars&, bool) {
    ++*launches;
    if (P.nseg <= SMALL_SEG) return launch_ag_t<SMALL_SEG>(P, rep, master, st, stream);
    return launch_ag_t<BIG_SEG>(P, rep, master, st, stream);
  });
}

cudaError_t launch_repair(const Plan& P0, uint16_t* const* rep, float* const* master2, const dp_step_state_t* st,
                          cudaStream_t stream, uint64_t* launches) {
  StepScalars s0{};
  return for_each_chunk(P0, s0, [&](const Plan& P, const StepScalars&, bool) {
    ++*launches;
    if (P.nseg <= SMALL_SEG) return launch_repair_t<SMALL_SEG>(P, rep, master2, st, stream);
    return launch_repair_t<BIG_SEG>(P, rep, master2, st, stream);
  });
}

cudaError_t launch_commit(dp_step_state_t* st, double b1, double b2, const ScalerK& scaler, int flip_set,
                          cudaStream_t stream, uint64_t* launches) {
  ++*launches;
  commit_kernel<<<1, 1, 0, stream>>>(st, b1, b2, scaler, flip_set);
  return cudaGetLastError();
}

cudaError_t launch_state_init(dp_step_state_t* st, cudaStream_t stream, uint64_t* launches) {
  ++*launches;
  state_init_kernel<<<1, 1, 0, stream>>>(st);
  return cudaGetLastError();
}

cudaError_t launch_scaler_init(dp_step_state_t* st, float scale, cudaStream_t stream, uint64_t* launches) {
  ++*launches;
  scaler_init_kernel<<<1, 1, 0, stream>>>(st, scale);
  return cudaGetLastError();
}

cudaError_t launch_selftest_wait(dp_step_state_t* st, uint64_t timeout_ns, cudaStream_t stream, uint64_t* launches) {
  ++*launches;
  selftest_wait_kernel<<<1, 32, 0, stream>>>(st, timeout_ns);
  return cudaGetLastError();
}

}  // namespace dp
