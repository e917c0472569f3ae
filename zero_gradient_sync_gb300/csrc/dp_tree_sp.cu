// The tree reduction order's single pass (sm_103a): pass A in tree order and the update in one launch, with
// the optimizer state double-buffered as in the ring order's single pass.
//
// The sum is the binomial tree of dp_tree.cu ("Data vs Tensor vs Pipeline Parallelism", DP gradient sync at
// scale: NCCL's tree beside the ring), computed the rank-major way in groups of G ranks (G = 4 for n >= 3):
// a stage holds micro-step k of every rank of a group for one sub-tile; each consumer thread carries the
// group's leaf sums across the micro-steps and adds them up the group's tree (levels 0 and 1, which pair
// ranks only inside aligned blocks of four).  The group totals then join as the tree's levels 2 and 3 do:
// groups 0 and 1, groups 2 and 3, then the two halves, each time the lower block on the left.  Each leaf is
// the same chain and each merge the same operation on the same operands as in the two-pass tree kernel, so
// gbar -- and with it the whole step -- is the same bits.  One instance serves every rank count of its class:
// the leaves are registers indexed at compile time, and the group size only switches merges and loads on or
// off.  Groups of four keep the leaves to 32 registers beside the update's working set.
//
// Per tile the sub-tiles' gbar goes into a shared tile; then the single pass's per-tile steps take over
// (dp_single.cuh): the tile's old master/m/v, bulk-copied into shared memory by the producer while the
// gradients stream, Adam into the other state set, and the all-gather of the bf16 image into the replicas.
// The shared-memory layout is the ring order's shared-gbar single pass -- 90 KB of stages (here six of
// 15 KB), the gbar tile, the bf16 staging tile and the state tile -- with room for six barrier pairs.

#include "dp_device.cuh"
#include "dp_internal.h"
#include "dp_launch.h"
#include "dp_single.cuh"

namespace dp {
namespace {

constexpr int TS_SLOT = RA_IN_BYTES;                          // 15 KB a stage
constexpr int TS_NST = ra_stages<1>() * RA_STAGE_BYTES / TS_SLOT;  // six stages in the shared-gbar pass's 90 KB
constexpr int TS_SMEM = ra_bar_offset<1>() + 2 * TS_NST * 8 + 16 + 32;
static_assert(TS_NST * TS_SLOT == ra_stages<1>() * RA_STAGE_BYTES, "the stages end where the gbar tile starts");
static_assert(TS_SMEM + 1024 <= 227 * 1024, "shared memory fits one CTA");
// Element classes: EPT elements a thread per sub-tile, groups of G = 16 / EPT ranks -- EPT 16 for n = 1, 8 for
// n = 2, 4 for n >= 3 -- so a group's stage is one 15 KB slot and its leaves 8 packed lanes.
template <int EPT>
__host__ __device__ constexpr int ts_g() { return 16 / EPT; }
template <int EPT>
__host__ __device__ constexpr int ts_sub() { return RA_CTHREADS * EPT; }
template <int EPT>
__host__ __device__ constexpr int ts_in_bytes() { return 2 * ts_sub<EPT>(); }
static_assert(ts_g<16>() * ts_in_bytes<16>() == TS_SLOT && ts_g<8>() * ts_in_bytes<8>() == TS_SLOT &&
                  ts_g<4>() * ts_in_bytes<4>() == TS_SLOT,
              "a group's stage fills one slot");
static_assert(TILE % ts_sub<4>() == 0 && TILE % ts_sub<8>() == 0 && TILE == ts_sub<16>(),
              "a tile is a whole number of sub-tiles");
static_assert(ts_in_bytes<4>() % 16 == 0, "sub-tiles start on 16-byte boundaries");
static_assert(DP_MAX_N <= 4 * ts_g<4>(), "four groups of four cover every rank count");

// The elements [lo, hi) of a tile inside sub-tile h of its cell, copied as the 8-aligned hull
// [lo & ~7, min(ceil8(hi), psi & ~7)); the producer stores the buffer's last partial 8-group after it.
struct SubRange {
  int64_t lo, hi, sa;
  __device__ __forceinline__ bool empty() const { return lo >= hi; }
};
__device__ __forceinline__ SubRange sub_range(const Tile& t, int h, int sub) {
  const int64_t cb = (t.start / TILE) * TILE + (int64_t)h * sub;
  SubRange x;
  x.lo = t.start > cb ? t.start : cb;
  x.hi = t.end < cb + sub ? t.end : cb + sub;
  x.sa = x.lo & ~int64_t(7);
  return x;
}

// EPT bf16 (EPT / 2 words) from shared memory: one 8- or 16-byte load, or two 16-byte loads.
template <int EPT>
__device__ __forceinline__ void ts_load(const unsigned char* s, uint32_t (&w)[EPT / 2]) {
  if constexpr (EPT == 4) {
    const uint2 v = *reinterpret_cast<const uint2*>(s);
    w[0] = v.x; w[1] = v.y;
  } else {
#pragma unroll
    for (int c = 0; c < EPT / 8; ++c) {
      const uint4 v = *reinterpret_cast<const uint4*>(s + 16 * c);
      w[4 * c + 0] = v.x; w[4 * c + 1] = v.y; w[4 * c + 2] = v.z; w[4 * c + 3] = v.w;
    }
  }
}

// left + right on W packed lanes, the lower-index block on the left.  Compensated: (H, e) = TwoSum(H_l, H_r),
// L = (L_l + e) + L_r; plain: H = H_l + H_r.
template <bool COMP, int W>
__device__ __forceinline__ void ts_merge(f2_t (&hl)[W], f2_t (&ll)[W], const f2_t (&hr)[W], const f2_t (&lr)[W]) {
#pragma unroll
  for (int u = 0; u < W; ++u) {
    if constexpr (COMP) {
      f2_t e;
      const f2_t H = f2_two_sum(hl[u], hr[u], e);
      ll[u] = f2_add(f2_add(ll[u], e), lr[u]);
      hl[u] = H;
    } else {
      hl[u] = f2_add(hl[u], hr[u]);
    }
  }
}

// One micro-step of the group's first ng ranks into their leaves: the first sets h = x (l = 0), later ones
// (h, e) = TwoSum(h, x), l = l + e (plain: h = h + x).
template <bool COMP, int MAXG, int W, bool FIRST>
__device__ __forceinline__ void ts_fold(f2_t (&h)[MAXG][W], f2_t (&l)[MAXG][W], const uint32_t (&w)[MAXG][W], int ng) {
#pragma unroll
  for (int r = 0; r < MAXG; ++r) {
    if (r < ng) {
#pragma unroll
      for (int u = 0; u < W; ++u) {
        const f2_t x = bf16x2_to_f2(w[r][u]);
        if (FIRST) {
          h[r][u] = x;
          if constexpr (COMP) l[r][u] = 0ull;
        } else if constexpr (COMP) {
          f2_t e;
          h[r][u] = f2_two_sum(h[r][u], x, e);
          l[r][u] = f2_add(l[r][u], e);
        } else {
          h[r][u] = f2_add(h[r][u], x);
        }
      }
    }
  }
}

// The binomial tree over the group's first ng leaves, levels 1 and 2 apart: block r takes block r + STEP on
// its right when that block exists; the total is left in leaf 0.
template <bool COMP, int MAXG, int W, int STEP>
__device__ __forceinline__ void ts_level(f2_t (&h)[MAXG][W], f2_t (&l)[MAXG][W], int ng) {
#pragma unroll
  for (int r = 0; r + STEP < MAXG; r += 2 * STEP)
    if (r + STEP < ng) ts_merge<COMP, W>(h[r], l[r], h[r + STEP], l[r + STEP]);
}
template <bool COMP, int MAXG, int W>
__device__ __forceinline__ void ts_tree(f2_t (&h)[MAXG][W], f2_t (&l)[MAXG][W], int ng) {
  if constexpr (MAXG > 1) ts_level<COMP, MAXG, W, 1>(h, l, ng);
  if constexpr (MAXG > 2) ts_level<COMP, MAXG, W, 2>(h, l, ng);
  static_assert(MAXG <= 4, "a group has at most four ranks");
}

template <int MAXSEG, bool COMP, int EPT>
__global__ void __launch_bounds__(RA_THREADS, 1) tree_single_kernel(const __grid_constant__ ReduceParams<MAXSEG> p) {
  constexpr int NST = TS_NST;
  constexpr int MAXG = ts_g<EPT>();
  constexpr int W = EPT / 2;
  constexpr int SUB = ts_sub<EPT>();
  constexpr int IN = ts_in_bytes<EPT>();
  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char* stages = smem;
  float* s_g = reinterpret_cast<float*>(smem + NST * TS_SLOT);
  uint16_t* s_stage = reinterpret_cast<uint16_t*>(smem + NST * TS_SLOT + ra_gbar_bytes<1>());
  float* s_state = reinterpret_cast<float*>(smem + NST * TS_SLOT + ra_gbar_bytes<1>() + TILE * 2);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + ra_bar_offset<1>());
  uint64_t* empty = full + NST;
  uint64_t* sfull = empty + NST;        // the tile's state has landed (producer + bytes)
  uint64_t* sempty = sfull + 1;         // the update is done reading it (consumer warps)
  volatile int* s_abort = reinterpret_cast<volatile int*>(sfull + 2);
  unsigned long long* s_count = reinterpret_cast<unsigned long long*>(sfull + 3);
  __shared__ float s_inv;
  __shared__ float s_k[2];
  __shared__ int s_cur;
  __shared__ int s_ragged_buf[2];       // the current tile's head / tail state groups are in s_state
  volatile int* s_ragged = s_ragged_buf;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n = p.n, a = p.a;
  const int ngroups = (n + MAXG - 1) / MAXG;
  const int ntiles = p.seg.ntiles;
  const int64_t psi = p.seg.psi;
  const int64_t p8 = psi & ~int64_t(7);

  if (tid == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), RA_CWARPS);
    }
    mbar_init(smem_u32(sfull), 1);
    mbar_init(smem_u32(sempty), RA_CWARPS);
    *s_abort = 0;
    *s_count = 0ull;
    float inv = p.inv;
    if (p.scaler.enabled) {
      // fl32(1 / (n S)) from the device-resident scale, as for the ring order.
      const float sc = *reinterpret_cast<volatile const float*>(&p.state->loss_scale);
      inv = (float)(1.0 / ((double)p.n * (double)sc));
      if (!(sc > 0.0f) || nonfinite(sc) || !(inv >= 1.17549435e-38f) || nonfinite(inv)) {
        record_error(p.state, DP_ERR_INVALID_ARG);
        *s_abort = 1;
        inv = 0.0f;
      }
    }
    s_inv = inv;
    // Bias corrections of the step being taken (t + 1): the same double products the finish stores.
    const volatile dp_step_state_t* vs = p.state;
    s_k[0] = (float)((double)p.lr / (1.0 - vs->b1t * p.beta1));
    s_k[1] = (float)(1.0 / sqrt(1.0 - vs->b2t * p.beta2));
    s_cur = (int)(vs->cur_set & 1u);
    fence_mbar_init();
  }
  __syncthreads();

  unsigned bad = 0;
  if (warp == RA_CWARPS) {
    // ------------------------------------------------------------ producer warp: per sub-tile and group, micro-step
    // k of the group's ranks (lane 0 waits for the slot and posts the byte count, lane r copies rank r); the
    // tile's old state once the tile's first NST stages are issued.
    RingPos<NST> rp;
    TileWalker<MAXSEG> walk;
    uint32_t sit = 0;
    bool stop = false;
    for (int tile = blockIdx.x; tile < ntiles && !stop; tile += gridDim.x) {
      const Tile t = walk.at(p.seg, tile);
      int subs = 0;
      for (int h = 0; h < TILE / SUB; ++h) subs += sub_range(t, h, SUB).empty() ? 0 : 1;
      const int tile_stages = subs * ngroups * a;
      const int state_after = tile_stages < NST ? tile_stages : NST;
      int sq = 0;
      for (int h = 0; h < TILE / SUB && !stop; ++h) {
        const SubRange x = sub_range(t, h, SUB);
        if (x.empty()) continue;
        int64_t sb = (x.hi + 7) & ~int64_t(7);
        if (sb > p8) sb = p8;
        const uint32_t bytes = sb > x.sa ? (uint32_t)(sb - x.sa) * 2u : 0u;
        const bool tail = x.hi > p8;   // the sub-tile holds elements of the buffer's last partial 8-group
        for (int gq = 0; gq < ngroups && !stop; ++gq) {
          const int r0 = gq * MAXG, ng = n - r0 < MAXG ? n - r0 : MAXG;
          for (int k = 0; k < a; ++k) {
            const uint32_t fb = smem_u32(&full[rp.slot]);
            int ok = 1;
            if (lane == 0) {
              if (*s_abort) {
                ok = 0;
              } else if (rp.count >= (uint32_t)NST &&
                         !mbar_wait_bounded(smem_u32(&empty[rp.slot]), rp.phase ^ 1u, p.timeout_ns, s_abort)) {
                if (!*s_abort) record_error(p.state, DP_ERR_TIMEOUT);
                *s_abort = 1;
                ok = 0;
              }
            }
            ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
            __syncwarp();
            if (!ok) {
              stop = true;
              break;
            }
            unsigned char* slot = stages + rp.slot * TS_SLOT;
            if (tail && lane < ng) {
              // The buffer's last partial 8-group (zeros past psi), stored by this lane; ordered before the async
              // proxy's later writes into the slot by the fence, and before the consumers' reads by the arrive.
              const uint16_t* src = p.g[(r0 + lane) * a + k];
              uint32_t v[4];
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const uint32_t lo = p8 + 2 * u < psi ? (uint32_t)src[p8 + 2 * u] : 0u;
                const uint32_t hi = p8 + 2 * u + 1 < psi ? (uint32_t)src[p8 + 2 * u + 1] : 0u;
                v[u] = lo | (hi << 16);
              }
              *reinterpret_cast<uint4*>(slot + lane * IN + (p8 - x.sa) * 2) = make_uint4(v[0], v[1], v[2], v[3]);
              fence_proxy_async_smem();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive_expect_tx(fb, bytes * (uint32_t)ng);
            __syncwarp();
            if (bytes && lane < ng)
              bulk_g2s(smem_u32(slot + lane * IN), p.g[(r0 + lane) * a + k] + x.sa, bytes, fb);
            rp.next();
            if (++sq == state_after) {
              if (lane == 0) sp_issue_state(p, t, s_cur, sit, s_state, s_ragged, sfull, sempty, s_abort);
              __syncwarp();
            }
          }
        }
      }
    }
    if (lane == 0 && *s_abort) {
      // Never leave with copies in flight: the last state copy, then the newest issued phase of every slot.
      if (sit > 0) (void)mbar_wait_bounded(smem_u32(sfull), (sit - 1) & 1u, p.timeout_ns, nullptr);
      const uint32_t it = rp.count;
      const uint32_t first = it > (uint32_t)NST ? it - NST : 0u;
      for (uint32_t y = first; y < it; ++y)
        (void)mbar_wait_bounded(smem_u32(&full[y % NST]), (y / NST) & 1u, p.timeout_ns, nullptr);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ consumers
    const f2_t inv2 = f2_pack(s_inv, s_inv);
    RingPos<NST> rp;
    TileWalker<MAXSEG> walk;
    bool live = true;
    uint32_t sit_c = 0;   // tiles whose state this thread has used
    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
      const Tile t = walk.at(p.seg, tile);
      const int64_t cb = (t.start / TILE) * TILE;
      for (int h = 0; h < TILE / SUB; ++h) {
        const SubRange x = sub_range(t, h, SUB);
        if (x.empty()) continue;
        const int64_t e0 = x.sa + EPT * tid;
        const bool active = e0 < x.hi;

        // One stage (one micro-step of the group's ng ranks): wait for its bytes, take this thread's EPT values of
        // each rank, release the slot.  Every value comes from shared memory: the producer stored the buffer's
        // last partial 8-group there too.  A thread past the sub-tile's end reads bytes it never uses.
        auto take = [&](int ng, auto& w) {
          if (live && !mbar_wait_bounded(smem_u32(&full[rp.slot]), rp.phase, p.timeout_ns, s_abort)) {
            if (!*s_abort) record_error(p.state, DP_ERR_TIMEOUT);
            *s_abort = 1;
            live = false;
          }
          const unsigned char* src_s = stages + rp.slot * TS_SLOT + 2 * EPT * tid;
#pragma unroll
          for (int r = 0; r < MAXG; ++r)
            if (r < ng) ts_load<EPT>(src_s + r * IN, w[r]);
          // The slot is refilled by the async proxy: order this thread's reads of it before that write.
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&empty[rp.slot]));
          rp.next();
        };
        // A group's leaves over the micro-steps, then its tree; the total is left in leaf 0.
        auto group = [&](int ng, auto& hs, auto& ls) {
          {
            uint32_t w[MAXG][W];
            take(ng, w);
            ts_fold<COMP, MAXG, W, true>(hs, ls, w, ng);
          }
          for (int k = 1; k < a; ++k) {
            uint32_t w[MAXG][W];
            take(ng, w);
            ts_fold<COMP, MAXG, W, false>(hs, ls, w, ng);
          }
          ts_tree<COMP, MAXG, W>(hs, ls, ng);
        };

        // Group by group: its total joins the others as the tree's levels 2 and 3 do -- A holds ranks [0, 8),
        // B ranks [8, 16), and B joins A on the right at the end.  With n <= 2 there is one group and A is its
        // total.
        f2_t Ah[W], Al[W];
        if constexpr (MAXG < 4) {
          f2_t hs[MAXG][W], ls[MAXG][W];
          group(n, hs, ls);
#pragma unroll
          for (int u = 0; u < W; ++u) {
            Ah[u] = hs[0][u];
            if constexpr (COMP) Al[u] = ls[0][u];
          }
        } else {
          f2_t Bh[W], Bl[W];
          for (int gq = 0; gq < ngroups; ++gq) {
            const int r0 = gq * MAXG, ng = n - r0 < MAXG ? n - r0 : MAXG;
            f2_t hs[MAXG][W], ls[MAXG][W];
            group(ng, hs, ls);
            if (gq == 0 || gq == 2) {
#pragma unroll
              for (int u = 0; u < W; ++u) {
                if (gq == 0) {
                  Ah[u] = hs[0][u];
                  if constexpr (COMP) Al[u] = ls[0][u];
                } else {
                  Bh[u] = hs[0][u];
                  if constexpr (COMP) Bl[u] = ls[0][u];
                }
              }
            } else if (gq == 1) {
              ts_merge<COMP, W>(Ah, Al, hs[0], ls[0]);
            } else {
              ts_merge<COMP, W>(Bh, Bl, hs[0], ls[0]);
            }
          }
          if (ngroups > 2) ts_merge<COMP, W>(Ah, Al, Bh, Bl);
        }

        // gbar = fl(p * inv) into the tile's shared gbar (indexed by global position in the cell); count the
        // non-finite ones of this tile.
        float o[EPT];
#pragma unroll
        for (int u = 0; u < W; ++u) {
          const f2_t pp = COMP ? f2_add(Ah[u], Al[u]) : Ah[u];
          f2_unpack(f2_mul(pp, inv2), o[2 * u], o[2 * u + 1]);
        }
        if (active) {
          float* gs = s_g + (e0 - cb);
          if (e0 >= x.lo && e0 + EPT <= x.hi) {
#pragma unroll
            for (int c = 0; c < EPT / 4; ++c)
              *reinterpret_cast<float4*>(gs + 4 * c) = make_float4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
#pragma unroll
            for (int u = 0; u < EPT; ++u) bad += nonfinite(o[u]);
          } else {
#pragma unroll
            for (int u = 0; u < EPT; ++u)
              if (e0 + u >= x.lo && e0 + u < x.hi) {
                gs[u] = o[u];
                bad += nonfinite(o[u]);
              }
          }
        }
      }

      // The tile's gbar is complete in s_g once every consumer thread is here; the previous tile's replica
      // stores must have read s_stage before the update rewrites it.
      if (tid == 0) bulk_wait_read<0>();
      named_bar_sync(1, RA_CTHREADS);
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
      fused_update(p, t, K, s_cur, s_g, s_stage, s_state, s_ragged, tid);
      // Order this thread's reads of s_state (and writes of s_stage) before the async proxy's next use of them,
      // then hand s_state back to the producer.
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(sempty));
      ++sit_c;
      named_bar_sync(1, RA_CTHREADS);
      // All-gather: the staged bf16 tile into every replica.
      sp_gather(p, t, cb, s_stage, n, tid);
    }
  }

  // ------------------------------------------------------------ CTA total, then the grid's
  unsigned long long c = bad;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) c += __shfl_xor_sync(0xFFFFFFFFu, c, off);
  __syncthreads();
  if (lane == 0 && c) atomicAdd(s_count, c);
  __syncthreads();
  if (tid == 0) bulk_wait_all();   // the last tile's replica stores
  if (tid == 0)
    finish_reduction(p.state, *s_count, (*s_count != 0ull) || *s_abort, p.advance, p.beta1, p.beta2, &p.scaler, 1,
                     p.merge);
}

template <int MAXSEG, bool COMP, int EPT>
cudaError_t launch_tree_single_t(const Plan& P, const uint16_t* const* g, int a, const StepScalars& s, int advance,
                                 dp_step_state_t* st, const FusedArgs& fa, cudaStream_t stream) {
  // A class below four ranks a group has exactly one group; groups of four cover up to 16 ranks.
  if (P.n < 1 || (ts_g<EPT>() < 4 ? P.n != ts_g<EPT>() : P.n > 4 * ts_g<EPT>())) return cudaErrorInvalidValue;
  ReduceParams<MAXSEG> prm;
  fill_reduce_params(prm, P, g, a, nullptr, s, advance, st, &fa);
  auto kern = tree_single_kernel<MAXSEG, COMP, EPT>;
  // The opt-in shared-memory size is set once per device (not inside a stream capture on later calls).
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, TS_SMEM);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  // Every CTA takes part in the grid-wide finish, so at least one CTA runs even with no tiles.
  int grid = sm_count();
  if (P.ntiles < grid) grid = P.ntiles > 0 ? P.ntiles : 1;
  kern<<<grid, RA_THREADS, TS_SMEM, stream>>>(prm);
  return cudaGetLastError();
}

// The element class of n ranks: one group of n for n <= 2 (16 elements a thread for n = 1, 8 for n = 2), else
// groups of four at 4 elements a thread.
constexpr int ts_ept_of(int n) { return n == 1 ? 16 : (n == 2 ? 8 : 4); }
static_assert(ts_g<ts_ept_of(1)>() == 1 && ts_g<ts_ept_of(2)>() == 2 && ts_g<ts_ept_of(3)>() == 4,
              "a class below four ranks a group holds its n in one group");

template <int MAXSEG, bool COMP>
cudaError_t launch_tree_single_c(const Plan& P, const uint16_t* const* g, int a, const StepScalars& s, int advance,
                                 dp_step_state_t* st, const FusedArgs& fa, cudaStream_t stream) {
  switch (ts_ept_of(P.n)) {
    case 16: return launch_tree_single_t<MAXSEG, COMP, 16>(P, g, a, s, advance, st, fa, stream);
    case 8: return launch_tree_single_t<MAXSEG, COMP, 8>(P, g, a, s, advance, st, fa, stream);
    default: return launch_tree_single_t<MAXSEG, COMP, 4>(P, g, a, s, advance, st, fa, stream);
  }
}

}  // namespace

cudaError_t launch_tree_single(const Plan& P, const uint16_t* const* g, int a, const StepScalars& s,
                               dp_step_state_t* st, const FusedArgs& fa, cudaStream_t stream) {
  const bool comp = s.mode == DP_SUM_COMPENSATED;
  const int adv = s.defer ? 0 : 1;
  if (P.nseg <= SMALL_SEG)
    return comp ? launch_tree_single_c<SMALL_SEG, true>(P, g, a, s, adv, st, fa, stream)
                : launch_tree_single_c<SMALL_SEG, false>(P, g, a, s, adv, st, fa, stream);
  return comp ? launch_tree_single_c<BIG_SEG, true>(P, g, a, s, adv, st, fa, stream)
              : launch_tree_single_c<BIG_SEG, false>(P, g, a, s, adv, st, fa, stream);
}

}  // namespace dp
